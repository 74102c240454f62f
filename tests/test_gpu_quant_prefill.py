"""GPU parity for Q4_0 / Q4_K prefill on the tensor cores (M >= 16).

Both formats are affine per 32 weights (Q4_0: scale d, bias -8d; Q4_K: scale
d*sc, bias -dmin*m), so these calls rewrite the weights as packed affine codes
in the workspace and run the affine tensor-core prefill. Bars, per output:
    |y - ref| <= 2e-3 * sum_k |x_k w_k| + 1e-6          (the prefill bar)
and, pinning the path's one approximation (x rounded to fp16 after a per-row
power-of-two scale), the oracle fed the rounded activations must match y to
the f32 bar (1e-5); for the folded-weight kernel the oracle also gets the
weights it multiplies (each row times a power of two, rounded to fp16). A
workspace too small for the repacked weights selects the CUDA-core path (f32
bar). The dual projection stays bitwise equal to two single projections.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, dev, to_dev
from test_gpu_prefill import REL_TC, _rounded_x, kernel, rounded_ref  # noqa: F401 (fixture)
from test_gpu_prefill import tensor_cores_from_m16  # noqa: F401 (autouse fixture)

pytestmark = pytest.mark.gpu


def _q4_0_rowbound(w, N, K):
    """max over the row's blocks of |d| * 15 + |8 d| (the repacked s, b)."""
    blk = np.asarray(w, np.uint8).reshape(N, K // 32, 18)
    d = oracle.half_to_float_array(blk[:, :, 0].astype(np.uint16) | (blk[:, :, 1].astype(np.uint16) << 8))
    return np.max(np.abs(d.astype(np.float32)) * np.float32(23.0), axis=1)


def _q4_k_rowbound(w, N, K):
    """max over the row's sub-blocks of |d sc| * 15 + |dmin m| (the repacked s, b)."""
    blk = np.asarray(w, np.uint8).reshape(N, K // 256, 144)
    d = oracle.half_to_float_array(blk[:, :, 0].astype(np.uint16) | (blk[:, :, 1].astype(np.uint16) << 8))
    dm = oracle.half_to_float_array(blk[:, :, 2].astype(np.uint16) | (blk[:, :, 3].astype(np.uint16) << 8))
    out = np.zeros(N, np.float32)
    for n in range(N):
        for sb in range(K // 256):
            for j in range(8):
                sc, m = oracle.q4_k_scale_min(blk[n, sb, 4:16], j)
                v = np.float32(abs(np.float32(d[n, sb]) * np.float32(sc))) * np.float32(15.0) \
                    + np.float32(abs(np.float32(dm[n, sb]) * np.float32(m)))
                out[n] = max(out[n], v)
    return out


def _rounding_check(y, kernel, w, x, M, N, K, fmt, what):
    if fmt == "q4_0":
        if kernel:
            ref, bound = oracle.gemv_q4_0(w, _rounded_x(x), M, N, K)
        else:
            ref, bound = rounded_ref(x, oracle.dequant_q4_0(w, N, K), _q4_0_rowbound(w, N, K), M, N, K)
    else:
        if kernel:
            ref, bound = oracle.gemv_q4_k(w, _rounded_x(x), M, N, K)
        else:
            ref, bound = rounded_ref(x, oracle.dequant_q4_k(w, N, K), _q4_k_rowbound(w, N, K), M, N, K)
    assert_parity(y, ref, bound, what=what)


def _ws(op, M, N, K):
    n = qg.workspace_size(op, M, N, K)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=dev())


@pytest.mark.parametrize("M,N,K", [(16, 100, 256), (37, 130, 1024), (200, 257, 4096)])
def test_q4_0_prefill(M, N, K, kernel):
    c = synth.q4_0_case(4000 + M + N, N, K, M)
    ws = _ws(qg.QG_OP_Q4_0, M, N, K)
    assert ws.numel() > N * K // 2  # room for the repacked weights
    y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(c["x"]), N=N, workspace=ws)
    ref, bound = oracle.gemv_q4_0(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, rel=REL_TC, what=f"q4_0 prefill M={M} N={N} K={K}")
    _rounding_check(y, kernel, c["w"], c["x"], M, N, K, "q4_0", f"q4_0 prefill vs rounded operands M={M}")


@pytest.mark.parametrize("M,N,K", [(16, 70, 256), (64, 200, 4096)])
def test_dual_q4_0_prefill_equals_two_singles(M, N, K, kernel):
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
def test_q4_k_prefill(M, N, K, kernel):
    c = synth.q4_k_case(4200 + M + N, N, K, M)
    ws = _ws(qg.QG_OP_Q4_K, M, N, K)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N, workspace=ws)
    ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, rel=REL_TC, what=f"q4_k prefill M={M} N={N} K={K}")
    _rounding_check(y, kernel, c["w"], c["x"], M, N, K, "q4_k", f"q4_k prefill vs rounded operands M={M}")


def test_small_workspace_takes_cuda_cores():
    """With only the CUDA-core workspace the call stays on CUDA cores (f32 bar)."""
    M, N, K = 32, 96, 1024
    c = synth.q4_0_case(4300, N, K, M)
    small = torch.empty(16, dtype=torch.uint8, device=dev())
    y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(c["x"]), N=N, workspace=small)
    ref, bound = oracle.gemv_q4_0(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what="q4_0 M=32 on CUDA cores")


def test_prefill_integer_closed_form_q4_0(kernel):
    """d = 1 and x in {-1, 0, 1}: every value either kernel forms is an
    integer (x scaled by 2^14, weights q - 8 scaled by 2^10 in the folded
    kernel, all exact in fp16) small enough for f32 (at most
    K * 8 * 2^14 = 2^24 for K = 128 with exact codes), so y must be exact."""
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
