"""GPU parity for 8 < M < 64 on the CUDA cores (the default for every M below
QG_OPT_PREFILL_MIN_M = 64), at the f32 bar of every GEMV test: per output
|y - ref| <= 1e-5 * sum_k |x_k w_k| + 1e-6 against the oracle. Every format:
Q4_0 single and dual (bitwise equal to two singles), Q4_K, and affine with
one code per byte and packed (bitwise equal), with M values on either side of
the old tensor-core threshold (16) and of the 8-row slices the kernels use.
"""
import numpy as np
import pytest

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, to_dev

pytestmark = pytest.mark.gpu

MS = [9, 12, 15, 16, 24, 33, 48, 63]


def test_default_threshold_keeps_mid_m_on_cuda_cores():
    assert qg.get_option(qg.QG_OPT_PREFILL_MIN_M) == 64


@pytest.mark.parametrize("M", MS)
def test_mid_m_q4_0_dual(M):
    N, K = 72, 1024
    c = synth.q4_0_case(7000 + M, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    assert_bitwise(ya, qg.qgemv_q4_0(wa, x, N=N), f"M={M} dual vs single")
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, what=f"q4_0 y_a M={M}")
    assert_parity(yb, rb, bb, what=f"q4_0 y_b M={M}")


@pytest.mark.parametrize("M", MS)
def test_mid_m_q4_k(M):
    N, K = 40, 2048
    c = synth.q4_k_case(7100 + M, N, K, M)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
    assert_parity(y, *oracle.gemv_q4_k(c["w"], c["x"], M, N, K), what=f"q4_k M={M}")


@pytest.mark.parametrize("M", MS)
def test_mid_m_affine(M):
    N, K, gs = 50, 1024, 64
    c = synth.affine_case(7200 + M, N, K, M, gs)
    x, s, b = to_dev(c["x"]), to_dev(c["s"]), to_dev(c["b"])
    yu = qg.qmm_affine(x, to_dev(c["q"]), s, b, gs, 0)
    yp = qg.qmm_affine(x, to_dev(c["q_packed"]), s, b, gs, 1)
    assert_bitwise(yp, yu, f"M={M} packed vs u8")
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(yu, ref, bound, what=f"affine M={M}")


@pytest.mark.parametrize("M", [16, 32])
def test_mid_m_full_width(M):
    """The sweep's mid-M shapes (N = K = 4096) on sampled rows."""
    N = K = 4096
    c = synth.q4_0_case(7300 + M, N, K, M, dual=True)
    ya, yb = qg.qgemv_dual_q4_0(to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"]), N=N)
    rows = np.arange(0, N, 61)
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K, rows=rows)
    assert_parity(ya.cpu().numpy()[:, rows], ra[:, rows], ba[:, rows], what=f"full width y_a M={M}")
    assert_parity(yb.cpu().numpy()[:, rows], rb[:, rows], bb[:, rows], what=f"full width y_b M={M}")
