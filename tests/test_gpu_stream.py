"""GPU parity of the streaming GEMV kernel (calls with M <= 2, K % 1024 == 0).

The same tolerance as the other GEMV tests (per output, |y - ref| <=
1e-5 * sum_k |x_k w_k| + 1e-6 against the oracle's f64 reference). Covered
here: every lanes-per-row width (K = 1024, 2048, 4096, 8192) and several steps
per row (K = 3072, 12288), ragged row counts, M = 1 and 2, affine group sizes
32..1024, both code storages (bitwise equal), ring shapes from one warp with two
slots to eight warps with eight, extreme and all-zero activations (the kernel
scales x by a power of two chosen from max|x|), and agreement with the staged
kernel it replaces (QG_OPT_STREAM = 0).
"""
import numpy as np
import pytest

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def stream_opts():
    """Every eligible call takes the streaming kernel here (the register-resident-x
    kernel, which would take most of them first, is switched off); the options
    are restored afterwards."""
    qg.set_option(qg.QG_OPT_STREAM, 2)
    qg.set_option(qg.QG_OPT_XREG, 0)
    yield
    qg.set_option(qg.QG_OPT_XREG, 1)
    qg.set_option(qg.QG_OPT_STREAM, 1)
    qg.set_option(qg.QG_OPT_STREAM_WARPS, 0)
    qg.set_option(qg.QG_OPT_STREAM_SLOTS, 0)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(37, 1024), (61, 2048), (45, 3072), (70, 4096), (19, 8192),
                                 (23, 12288)])
def test_stream_q4_0_dual(M, N, K):
    c = synth.q4_0_case(3000 + M * 13 + N, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    sa = qg.qgemv_q4_0(wa, x, N=N)
    assert_bitwise(ya, sa, f"stream dual vs single M={M} N={N} K={K}")
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, what=f"stream q4_0 y_a M={M} N={N} K={K}")
    assert_parity(yb, rb, bb, what=f"stream q4_0 y_b M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(29, 1024), (50, 4096), (21, 12288), (33, 8192)])
def test_stream_q4_k(M, N, K):
    c = synth.q4_k_case(3100 + M + N, N, K, M)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
    ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what=f"stream q4_k M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K,gs", [(37, 1024, 32), (64, 4096, 64), (20, 2048, 128),
                                    (17, 4096, 256), (25, 3072, 512), (16, 8192, 1024)])
def test_stream_affine(M, N, K, gs):
    c = synth.affine_case(3200 + M + N + gs, N, K, M, gs)
    x, s, b = to_dev(c["x"]), to_dev(c["s"]), to_dev(c["b"])
    yu = qg.qmm_affine(x, to_dev(c["q"]), s, b, gs, 0)
    yp = qg.qmm_affine(x, to_dev(c["q_packed"]), s, b, gs, 1)
    assert_bitwise(yp, yu, f"stream packed vs u8 M={M} N={N} K={K} gs={gs}")
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(yu, ref, bound, what=f"stream affine M={M} N={N} K={K} gs={gs}")


@pytest.mark.parametrize("warps,slots", [(1, 2), (2, 3), (3, 2), (8, 2), (8, 4), (6, 8)])
def test_stream_ring_shapes(warps, slots):
    M, N, K = 1, 301, 4096
    c = synth.q4_0_case(3300 + warps * 10 + slots, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    base = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    qg.set_option(qg.QG_OPT_STREAM_WARPS, warps)
    qg.set_option(qg.QG_OPT_STREAM_SLOTS, slots)
    ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    # The ring shape never changes the arithmetic.
    assert_bitwise(ya, base[0], f"ring {warps}x{slots} y_a")
    assert_bitwise(yb, base[1], f"ring {warps}x{slots} y_b")
    ck = synth.q4_k_case(3350 + warps, 77, 12288, 2)
    y = qg.qgemv_q4_k(to_dev(ck["w"]), to_dev(ck["x"]), N=77)
    ref, bound = oracle.gemv_q4_k(ck["w"], ck["x"], 2, 77, 12288)
    assert_parity(y, ref, bound, what=f"ring {warps}x{slots} q4_k")


@pytest.mark.parametrize("scale", [1e30, 3e-30, 1e-42, 0.0])
def test_stream_activation_magnitudes(scale):
    M, N, K, gs = 2, 40, 4096, 64
    c = synth.q4_0_case(3400, N, K, M)
    x = (c["x"].astype(np.float64) * scale).astype(np.float32)
    y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(x), N=N)
    ref, bound = oracle.gemv_q4_0(c["w"], x, M, N, K)
    assert np.isfinite(y.cpu().numpy()).all()
    assert_parity(y, ref, bound, what=f"q4_0 x*{scale}")
    a = synth.affine_case(3401, N, K, M, gs)
    xa = (a["x"].astype(np.float64) * scale).astype(np.float32)
    ya = qg.qmm_affine(to_dev(xa), to_dev(a["q_packed"]), to_dev(a["s"]), to_dev(a["b"]), gs, 1)
    ref, bound = oracle.qmm_affine(xa, a["q"], a["s"], a["b"], M, N, K, gs, False)
    assert_parity(ya, ref, bound, what=f"affine x*{scale}")


def test_stream_mixed_magnitudes():
    # One huge activation next to tiny ones in the same row.
    M, N, K = 1, 33, 4096
    c = synth.q4_k_case(3500, N, K, M)
    x = c["x"].copy()
    x[0, 7] = 3.0e37
    x[0, 100:200] *= np.float32(1e-35)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(x), N=N)
    ref, bound = oracle.gemv_q4_k(c["w"], x, M, N, K)
    assert_parity(y, ref, bound, what="q4_k mixed magnitudes")


@pytest.mark.parametrize("fmt", ["q4_0", "q4_k", "packed"])
def test_stream_matches_staged_kernel(fmt):
    M, N, K = 1, 260, 4096
    if fmt == "q4_0":
        c = synth.q4_0_case(3600, N, K, M)
        run = lambda: qg.qgemv_q4_0(to_dev(c["w"]), to_dev(c["x"]), N=N)
        ref, bound = oracle.gemv_q4_0(c["w"], c["x"], M, N, K)
    elif fmt == "q4_k":
        c = synth.q4_k_case(3601, N, K, M)
        run = lambda: qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
        ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    else:
        c = synth.affine_case(3602, N, K, M, 64)
        run = lambda: qg.qmm_affine(to_dev(c["x"]), to_dev(c["q_packed"]), to_dev(c["s"]),
                                    to_dev(c["b"]), 64, 1)
        ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, 64, False)
    y1 = run()
    qg.set_option(qg.QG_OPT_STREAM, 0)
    y0 = run()
    assert_parity(y1, ref, bound, what=f"{fmt} stream")
    assert_parity(y0, ref, bound, what=f"{fmt} staged")


def test_stream_rows_of_different_magnitude():
    # M = 2 in one launch: each input row gets its own power-of-two scaling.
    M, N, K = 2, 48, 4096
    c = synth.q4_0_case(3700, N, K, M, dual=True)
    x = c["x"].copy()
    x[0] *= np.float32(1e35)
    x[1] *= np.float32(1e-20)
    ya, yb = qg.qgemv_dual_q4_0(to_dev(c["w"]), to_dev(c["w_b"]), to_dev(x), N=N)
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], x, M, N, K)
    assert_parity(ya, ra, ba, what="y_a rows of different magnitude")
    assert_parity(yb, rb, bb, what="y_b rows of different magnitude")
