"""GPU parity for the dequantize-fused GEMV family against the oracle.

Tolerance (written here, per output): |y - ref| <= 1e-5 * sum_k |x_k w_k| + 1e-6
with ref and the sum computed by the oracle in f64. Shapes span several row
chunks and a ragged tail, both kernel paths (16-byte-aligned rows and the
general kernel), every M bucket, the split-K path, and the full workload
sizes in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["default kernels", "staged kernel"])
def kernel_choice(request):
    """Every test here runs twice: with the library's default choice (the
    register-resident-x kernel for M <= 8 where it applies) and with that
    kernel switched off, so that the staged kernel keeps its coverage."""
    qg.set_option(qg.QG_OPT_XREG, 0 if request.param == "staged kernel" else 1)
    yield request.param
    qg.set_option(qg.QG_OPT_XREG, 1)


def _q4_0(case_id, M, N, K, dual=False, w_offset=0):
    c = synth.q4_0_case(case_id, N, K, M, dual=dual)
    d = {"w": to_dev(c["w"], w_offset), "x": to_dev(c["x"])}
    if dual:
        d["w_b"] = to_dev(c["w_b"], w_offset)
    return c, d


# --------------------------------------------------------------------- Q4_0
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", [(37, 512), (8, 256), (129, 1024)])
def test_q4_0_fast_path(M, N, K):
    c, d = _q4_0(1000 + M * 7 + N, M, N, K)
    y = qg.qgemv_q4_0(d["w"], d["x"], N=N)
    ref, bound = oracle.gemv_q4_0(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what=f"q4_0 M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K,off", [(1, 19, 96, 0), (3, 40, 32, 0), (2, 33, 512, 2),
                                       (9, 17, 256, 0), (1, 5, 4096 + 32, 0)])
def test_q4_0_general_path(M, N, K, off):
    c, d = _q4_0(1100 + N, M, N, K, w_offset=off)
    y = qg.qgemv_q4_0(d["w"], d["x"], N=N)
    ref, bound = oracle.gemv_q4_0(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what=f"q4_0 general M={M} N={N} K={K} off={off}")


def test_q4_0_config0_full():
    M, N, K = 1, 1024, 1024
    c, d = _q4_0(0, M, N, K)
    y = qg.qgemv_q4_0(d["w"], d["x"], N=N)
    ref, bound = oracle.gemv_q4_0(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what="config 0")


def test_q4_0_integer_inputs_exact():
    # d = 1 and integer x in [-4, 4]: every partial sum is an integer below
    # 2^24, so the GPU result must be exact.
    rng = np.random.default_rng(12)
    M, N, K = 4, 64, 1024
    nb = K // 32
    q = rng.integers(0, 16, size=(N, nb, 32)).astype(np.uint8)
    w = synth.q4_0_from_parts(np.full((N, nb), 0x3C00, np.uint16), q)
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    y = qg.qgemv_q4_0(to_dev(w), to_dev(x), N=N)
    exact = (x.astype(np.int64) @ (q.reshape(N, K).astype(np.int64) - 8).T).astype(np.float32)
    assert_bitwise(y, exact, "integer closed form")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("N,K", [(37, 512), (300, 2048)])
def test_dual_bitwise_equals_two_singles(M, N, K):
    c, d = _q4_0(1200 + M + N, M, N, K, dual=True)
    ya, yb = qg.qgemv_dual_q4_0(d["w"], d["w_b"], d["x"], N=N)
    sa = qg.qgemv_q4_0(d["w"], d["x"], N=N)
    sb = qg.qgemv_q4_0(d["w_b"], d["x"], N=N)
    assert_bitwise(ya, sa, "y_a vs single")
    assert_bitwise(yb, sb, "y_b vs single")
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, what="y_a")
    assert_parity(yb, rb, bb, what="y_b")


@pytest.mark.parametrize("M", [1, 8])
def test_dual_config1_full(M):
    """The benchmark's workload: two Q4_0 weights N = K = 4096, M = 1 and 8."""
    N = K = 4096
    c, d = _q4_0(1, M, N, K, dual=True)
    ya, yb = qg.qgemv_dual_q4_0(d["w"], d["w_b"], d["x"], N=N)
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, what=f"config1 y_a M={M}")
    assert_parity(yb, rb, bb, what=f"config1 y_b M={M}")
    sa = qg.qgemv_q4_0(d["w"], d["x"], N=N)
    assert_bitwise(ya, sa, "config1 y_a vs single")


def test_dual_split_k_path():
    # M = 8, K = 12288 does not fit x in shared memory: split-K with workspace.
    M, N, K = 8, 96, 12288
    c, d = _q4_0(1300, M, N, K, dual=True)
    assert qg.workspace_size(qg.QG_OP_DUAL_Q4_0, M, N, K) > 0
    ya, yb = qg.qgemv_dual_q4_0(d["w"], d["w_b"], d["x"], N=N)
    sa = qg.qgemv_q4_0(d["w"], d["x"], N=N)
    assert_bitwise(ya, sa, "split-K dual vs single")
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, what="split-K y_a")
    assert_parity(yb, rb, bb, what="split-K y_b")


# --------------------------------------------------------------------- Q4_K
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("N,K", [(37, 256), (100, 1024), (9, 4096)])
def test_q4_k_fast_path(M, N, K):
    c = synth.q4_k_case(1400 + M + N, N, K, M)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
    ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what=f"q4_k M={M} N={N} K={K}")


def test_q4_k_general_path_unaligned():
    M, N, K = 2, 21, 512
    c = synth.q4_k_case(1500, N, K, M)
    y = qg.qgemv_q4_k(to_dev(c["w"], 4), to_dev(c["x"]), N=N)
    ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what="q4_k general")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_q4_k_ffn_down_split_k(M):
    M_, N, K = M, 64, 12288
    c = synth.q4_k_case(1600 + M, N, K, M_)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
    ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M_, N, K)
    assert_parity(y, ref, bound, what=f"q4_k K=12288 M={M}")


@pytest.mark.parametrize("N", [4096, 12288])
def test_q4_k_config2_full(N):
    M, K = 1, 4096
    c = synth.q4_k_case(2, N, K, M)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
    ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what=f"config2 N={N}")


# ------------------------------------------------------------------- affine
@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("N,K,gs", [(37, 256, 64), (64, 4096, 64), (20, 1024, 128),
                                    (33, 512, 32), (16, 2048, 1024), (12, 256, 8)])
def test_affine_packed_equals_u8_and_oracle(M, N, K, gs):
    c = synth.affine_case(1700 + M + N + gs, N, K, M, gs)
    x, s, b = to_dev(c["x"]), to_dev(c["s"]), to_dev(c["b"])
    yu = qg.qmm_affine(x, to_dev(c["q"]), s, b, gs, 0)
    yp = qg.qmm_affine(x, to_dev(c["q_packed"]), s, b, gs, 1)
    assert_bitwise(yp, yu, f"packed vs u8 M={M} N={N} K={K} gs={gs}")
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(yu, ref, bound, what=f"affine M={M} N={N} K={K} gs={gs}")


@pytest.mark.parametrize("packed", [0, 1])
@pytest.mark.parametrize("M,N,K,gs", [(2, 13, 64, 2), (5, 9, 96, 4), (1, 7, 200, 8)])
def test_affine_general_path(M, N, K, gs, packed):
    c = synth.affine_case(1800 + N, N, K, M, gs)
    q = c["q_packed"] if packed else c["q"]
    y = qg.qmm_affine(to_dev(c["x"]), to_dev(q), to_dev(c["s"]), to_dev(c["b"]), gs, packed)
    ref, bound = oracle.qmm_affine(c["x"], q, c["s"], c["b"], M, N, K, gs, bool(packed))
    assert_parity(y, ref, bound, what=f"affine general M={M} gs={gs} packed={packed}")


@pytest.mark.parametrize("M", [1, 8])
def test_affine_config3_full(M):
    N = K = 4096
    gs = 64
    c = synth.affine_case(3, N, K, M, gs)
    x, s, b = to_dev(c["x"]), to_dev(c["s"]), to_dev(c["b"])
    yu = qg.qmm_affine(x, to_dev(c["q"]), s, b, gs, 0)
    yp = qg.qmm_affine(x, to_dev(c["q_packed"]), s, b, gs, 1)
    assert_bitwise(yp, yu, "config3 packed vs u8")
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(yu, ref, bound, what=f"config3 M={M}")


def test_affine_equals_dequant_then_matmul():
    # The pages' composition check: fused qmm == dequantize, then f64 matmul.
    M, N, K, gs = 5, 9, 96 * 4, 32
    c = synth.affine_case(1900, N, K, M, gs)
    W = qg.dequant_affine(to_dev(c["q"]), to_dev(c["s"]), to_dev(c["b"]), N, K, gs, 0)
    y = qg.qmm_affine(to_dev(c["x"]), to_dev(c["q"]), to_dev(c["s"]), to_dev(c["b"]), gs, 0)
    Wd = W.cpu().numpy().astype(np.float64)
    comp = c["x"].astype(np.float64) @ Wd.T
    bound = np.abs(c["x"].astype(np.float64)) @ np.abs(Wd).T
    assert_parity(y, comp, bound, what="fused vs composed")


# ------------------------------------------------- programmatic dependent launch
@pytest.mark.parametrize("M", [1, 3, 8])
def test_pdl_chain_reads_previous_output(M):
    """With QG_OPT_PDL a call may start while the previous one drains; it must
    still see the previous call's y when that y is its x."""
    N = K = 1024
    c = synth.q4_0_case(2100 + M, N, K, M, dual=True)
    wa, wb = to_dev(c["w"]), to_dev(c["w_b"])
    ck = synth.q4_k_case(2200 + M, N, K, M)
    wk = to_dev(ck["w"])
    qg.set_option(qg.QG_OPT_PDL, 1)
    try:
        x0 = to_dev(c["x"])
        ya, yb = qg.qgemv_dual_q4_0(wa, wb, x0, N=N)   # x1 = ya
        y2 = qg.qgemv_q4_k(wk, ya, N=N)                 # x2 = y2
        y3 = qg.qgemv_q4_0(wb, y2, N=N)
        torch.cuda.synchronize()
    finally:
        qg.set_option(qg.QG_OPT_PDL, 0)
    # The oracle replays the chain on the GPU's own intermediate outputs, so
    # each stage is checked against exactly the input it was given.
    (ra, ba), _ = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, what="chain stage 1")
    r2, b2 = oracle.gemv_q4_k(ck["w"], ya.cpu().numpy(), M, N, K)
    assert_parity(y2, r2, b2, what="chain stage 2")
    r3, b3 = oracle.gemv_q4_0(c["w_b"], y2.cpu().numpy(), M, N, K)
    assert_parity(y3, r3, b3, what="chain stage 3")
    assert qg.device_error() == 0


def test_pdl_option_roundtrip():
    assert qg.get_option(qg.QG_OPT_PDL) == 0
    qg.set_option(qg.QG_OPT_PDL, 1)
    assert qg.get_option(qg.QG_OPT_PDL) == 1
    qg.set_option(qg.QG_OPT_PDL, 0)
    with pytest.raises(qg.QGError):
        qg.set_option(qg.QG_OPT_PDL, 5)


# ------------------------------------------------------------- error paths
def test_invalid_arguments_rejected_before_launch():
    x = torch.zeros((1, 64), device=dev())
    w = torch.zeros(2 * 18 * 4, dtype=torch.uint8, device=dev())
    y = torch.zeros((1, 4), device=dev())
    L = qg.lib()
    s = torch.cuda.current_stream().cuda_stream
    assert L.qgemv_q4_0(w.data_ptr(), x.data_ptr(), y.data_ptr(), 0, 4, 64, None, 0, s) == 1
    assert L.qgemv_q4_0(w.data_ptr(), x.data_ptr(), y.data_ptr(), 1, 4, 48, None, 0, s) == 1
    assert L.qgemv_q4_0(w.data_ptr(), x.data_ptr(), x.data_ptr(), 1, 4, 64, None, 0, s) == 1
    assert L.qgemv_q4_0(w.data_ptr(), x.data_ptr() + 2, y.data_ptr(), 1, 4, 64, None, 0, s) == 3
    assert L.qgemv_dual_q4_0(w.data_ptr(), w.data_ptr(), x.data_ptr(), y.data_ptr(),
                             y.data_ptr(), 1, 4, 64, None, 0, s) == 1
    sb = torch.zeros((4, 1), device=dev())
    assert L.qmm_affine(x.data_ptr(), w.data_ptr(), sb.data_ptr(), sb.data_ptr(), y.data_ptr(),
                        1, 4, 64, 5, 0, None, 0, s) == 1
    assert L.qmm_affine(x.data_ptr(), w.data_ptr(), sb.data_ptr(), sb.data_ptr(), y.data_ptr(),
                        1, 4, 64, 64, 2, None, 0, s) == 1
    assert qg.device_error() == 0


def test_split_k_requires_workspace():
    M, N, K = 8, 16, 12288
    c = synth.q4_0_case(1950, N, K, M)
    w, x = to_dev(c["w"]), to_dev(c["x"])
    y = torch.empty((M, N), device=dev())
    L = qg.lib()
    rc = L.qgemv_q4_0(w.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, K, None, 0,
                      torch.cuda.current_stream().cuda_stream)
    assert rc == qg.QG_ERR_WORKSPACE


def test_bounded_wait_reports_instead_of_hanging():
    assert qg.device_error(clear=True) == 0
    qg.selftest_wait_timeout(20_000_000)  # 20 ms
    code = qg.device_error(clear=True)
    assert code == 8, code
    assert qg.device_error() == 0


def test_no_device_error_left():
    assert qg.device_error() == 0


@pytest.fixture
def staged_m1():
    """M = 1 calls on the staged kernel (the register-resident-x kernel off)."""
    qg.set_option(qg.QG_OPT_XREG, 0)
    yield
    qg.set_option(qg.QG_OPT_XREG, 1)


@pytest.mark.parametrize("ahead", [0, 1, 3])
def test_stages_ahead_does_not_change_results(ahead, staged_m1):
    """QG_OPT_STAGES_AHEAD only changes when chunks are requested, never the
    arithmetic: results are bitwise equal to the default schedule."""
    M, N, K = 1, 700, 4096
    c = synth.q4_0_case(2300 + ahead, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    base = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    old = qg.get_option(qg.QG_OPT_STAGES_AHEAD)
    qg.set_option(qg.QG_OPT_STAGES_AHEAD, ahead)
    try:
        ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    finally:
        qg.set_option(qg.QG_OPT_STAGES_AHEAD, old)
    assert_bitwise(ya, base[0], f"ahead={ahead} y_a")
    assert_bitwise(yb, base[1], f"ahead={ahead} y_b")


def test_eight_warp_coresident_variant_is_bitwise_equal(staged_m1):
    """QG_OPT_STAGED_WARPS = 8 changes the CTA shape (and lets the next launch's
    CTA share the SM), never an output's arithmetic."""
    M, N, K = 1, 900, 4096
    c = synth.q4_0_case(2400, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    base = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    qg.set_option(qg.QG_OPT_STAGED_WARPS, 8)
    try:
        ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    finally:
        qg.set_option(qg.QG_OPT_STAGED_WARPS, 0)
    assert_bitwise(ya, base[0], "8-warp y_a")
    assert_bitwise(yb, base[1], "8-warp y_b")
