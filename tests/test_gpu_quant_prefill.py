"""GPU parity for Q4_0 / Q4_K prefill on the tensor cores (M >= 16).

Both formats are affine per 32 weights (Q4_0: scale d, bias -8d; Q4_K: scale
d*sc, bias -dmin*m), so these calls rewrite the weights as packed affine codes
in the workspace and run the affine tensor-core prefill. Bars, per output:
    |y - ref| <= 2e-3 * sum_k |x_k w_k| + 1e-6          (the prefill bar)
and, pinning the path's one approximation (x rounded to fp16 after a per-row
power-of-two scale), the oracle fed the rounded activations must match y to
the f32 bar (1e-5). A workspace too small for the repacked weights selects the
CUDA-core path (f32 bar). The dual projection stays bitwise equal to two
single projections.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, dev, to_dev
from test_gpu_prefill import REL_TC, _rounded_x

pytestmark = pytest.mark.gpu


def _ws(op, M, N, K):
    n = qg.workspace_size(op, M, N, K)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=dev())


@pytest.mark.parametrize("M,N,K", [(16, 100, 256), (37, 130, 1024), (200, 257, 4096)])
def test_q4_0_prefill(M, N, K):
    c = synth.q4_0_case(4000 + M + N, N, K, M)
    ws = _ws(qg.QG_OP_Q4_0, M, N, K)
    assert ws.numel() > N * K // 2  # room for the repacked weights
    y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(c["x"]), N=N, workspace=ws)
    ref, bound = oracle.gemv_q4_0(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, rel=REL_TC, what=f"q4_0 prefill M={M} N={N} K={K}")
    xr = _rounded_x(c["x"])
    ref_r, bound_r = oracle.gemv_q4_0(c["w"], xr, M, N, K)
    assert_parity(y, ref_r, bound_r, what=f"q4_0 prefill vs rounded x M={M}")


@pytest.mark.parametrize("M,N,K", [(16, 70, 256), (64, 200, 4096)])
def test_dual_q4_0_prefill_equals_two_singles(M, N, K):
    c = synth.q4_0_case(4100 + M, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    ws = _ws(qg.QG_OP_DUAL_Q4_0, M, N, K)
    ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N, workspace=ws)
    sa = qg.qgemv_q4_0(wa, x, N=N, workspace=ws)
    sb = qg.qgemv_q4_0(wb, x, N=N, workspace=ws)
    assert_bitwise(ya, sa, "prefill y_a vs single")
    assert_bitwise(yb, sb, "prefill y_b vs single")
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, rel=REL_TC, what="prefill y_a")
    assert_parity(yb, rb, bb, rel=REL_TC, what="prefill y_b")


@pytest.mark.parametrize("M,N,K", [(16, 90, 256), (128, 260, 4096), (300, 64, 12288)])
def test_q4_k_prefill(M, N, K):
    c = synth.q4_k_case(4200 + M + N, N, K, M)
    ws = _ws(qg.QG_OP_Q4_K, M, N, K)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N, workspace=ws)
    ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, rel=REL_TC, what=f"q4_k prefill M={M} N={N} K={K}")
    xr = _rounded_x(c["x"])
    ref_r, bound_r = oracle.gemv_q4_k(c["w"], xr, M, N, K)
    assert_parity(y, ref_r, bound_r, what=f"q4_k prefill vs rounded x M={M}")


def test_small_workspace_takes_cuda_cores():
    """With only the CUDA-core workspace the call stays on CUDA cores (f32 bar)."""
    M, N, K = 32, 96, 1024
    c = synth.q4_0_case(4300, N, K, M)
    small = torch.empty(16, dtype=torch.uint8, device=dev())
    y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(c["x"]), N=N, workspace=small)
    ref, bound = oracle.gemv_q4_0(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what="q4_0 M=32 on CUDA cores")


def test_prefill_integer_closed_form_q4_0():
    """d = 1 and x in {-1, 0, 1}: every value the path forms is an integer
    (x is scaled by 2^14 and exact in fp16) of magnitude at most
    K * 8 * 2^14 = 2^24 for K = 128, so the result must be exact."""
    rng = np.random.default_rng(44)
    M, N, K = 48, 64, 128
    nb = K // 32
    q = rng.integers(0, 16, size=(N, nb, 32)).astype(np.uint8)
    w = synth.q4_0_from_parts(np.full((N, nb), 0x3C00, np.uint16), q)
    x = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    ws = _ws(qg.QG_OP_Q4_0, M, N, K)
    y = qg.qgemv_q4_0(to_dev(w), to_dev(x), N=N, workspace=ws)
    exact = (x.astype(np.int64) @ (q.reshape(N, K).astype(np.int64) - 8).T).astype(np.float32)
    assert_bitwise(y, exact, "q4_0 prefill integer closed form")
