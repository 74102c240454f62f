"""GPU parity of the register-resident-x GEMV kernel (calls with M <= 2).

Same tolerance as every f32 GEMV test, per output:
|y - ref| <= 1e-5 * sum_k |x_k w_k| + 1e-6 against the oracle's f64 reference.
Covered: every format, M = 1 and 2, K from 256 to 16384 (one to sixteen warps
per row group, Q4_0 blocks of both parities, partly filled warps), ragged row
counts and chunks that straddle the two matrices of a dual call, the full
workload sizes, the dual projection bitwise equal to two single ones, packed
affine codes bitwise equal to one code per byte, an exact integer closed form,
activations spanning the f32 exponent range (the kernel scales x by one power
of two chosen from max|x|), non-finite x, and agreement with the older
CUDA-core kernels (QG_OPT_XREG = 0).
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, to_dev

pytestmark = pytest.mark.gpu

Q4_0_SHAPES = [(37, 256), (61, 1024), (45, 2048), (70, 3072), (300, 4096), (19, 8192),
               (23, 12288), (9, 16384)]


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", Q4_0_SHAPES)
def test_xreg_q4_0_dual_and_single(M, N, K):
    c = synth.q4_0_case(5000 + 7 * M + N, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    sa = qg.qgemv_q4_0(wa, x, N=N)
    sb = qg.qgemv_q4_0(wb, x, N=N)
    assert_bitwise(ya, sa, f"dual vs single y_a M={M} N={N} K={K}")
    assert_bitwise(yb, sb, f"dual vs single y_b M={M} N={N} K={K}")
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, what=f"q4_0 y_a M={M} N={N} K={K}")
    assert_parity(yb, rb, bb, what=f"q4_0 y_b M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(29, 256), (50, 1024), (33, 3072), (64, 4096), (21, 8192),
                                 (17, 12288), (11, 16384)])
def test_xreg_q4_k(M, N, K):
    c = synth.q4_k_case(5100 + M + N, N, K, M)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
    ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    assert_parity(y, ref, bound, what=f"q4_k M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K,gs", [(37, 1024, 32), (64, 4096, 64), (20, 2048, 128),
                                    (17, 4096, 256), (25, 8192, 512), (16, 4096, 1024),
                                    (13, 12288, 64)])
def test_xreg_affine_packed_equals_u8(M, N, K, gs):
    c = synth.affine_case(5200 + M + N + gs, N, K, M, gs)
    x, s, b = to_dev(c["x"]), to_dev(c["s"]), to_dev(c["b"])
    yu = qg.qmm_affine(x, to_dev(c["q"]), s, b, gs, 0)
    yp = qg.qmm_affine(x, to_dev(c["q_packed"]), s, b, gs, 1)
    assert_bitwise(yp, yu, f"packed vs u8 M={M} N={N} K={K} gs={gs}")
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(yu, ref, bound, what=f"affine M={M} N={N} K={K} gs={gs}")


def test_xreg_full_workloads():
    """The benchmark's M = 1 shapes at full size: config 0, config 1 (dual),
    config 2 (Q4_K N = 4096 and 12288, and the FFN down shape) and config 3."""
    c = synth.q4_0_case(0, 1024, 1024, 1)
    y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(c["x"]), N=1024)
    assert_parity(y, *oracle.gemv_q4_0(c["w"], c["x"], 1, 1024, 1024), what="config 0")
    c = synth.q4_0_case(1, 4096, 4096, 1, dual=True)
    ya, yb = qg.qgemv_dual_q4_0(to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"]), N=4096)
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], 1, 4096, 4096)
    assert_parity(ya, ra, ba, what="config 1 y_a")
    assert_parity(yb, rb, bb, what="config 1 y_b")
    for N, K in ((4096, 4096), (12288, 4096), (4096, 12288)):
        c = synth.q4_k_case(2, N, K, 1)
        y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
        assert_parity(y, *oracle.gemv_q4_k(c["w"], c["x"], 1, N, K), what=f"q4_k N={N} K={K}")
    c = synth.affine_case(3, 4096, 4096, 1, 64)
    for packed in (0, 1):
        q = c["q_packed"] if packed else c["q"]
        y = qg.qmm_affine(to_dev(c["x"]), to_dev(q), to_dev(c["s"]), to_dev(c["b"]), 64, packed)
        ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], 1, 4096, 4096, 64, False)
        assert_parity(y, ref, bound, what=f"config 3 packed={packed}")
    assert qg.device_error() == 0


@pytest.mark.parametrize("M", [1, 2])
def test_xreg_integer_inputs_exact(M):
    # d = 1 and integer x in [-4, 4]: every product and partial sum is an
    # integer times one power of two, below 2^24 of it: the result is exact.
    rng = np.random.default_rng(77 + M)
    N, K = 96, 4096
    nb = K // 32
    q = rng.integers(0, 16, size=(N, nb, 32)).astype(np.uint8)
    w = synth.q4_0_from_parts(np.full((N, nb), 0x3C00, np.uint16), q)
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    y = qg.qgemv_q4_0(to_dev(w), to_dev(x), N=N)
    exact = (x.astype(np.int64) @ (q.reshape(N, K).astype(np.int64) - 8).T).astype(np.float32)
    assert_bitwise(y, exact, "integer closed form")


@pytest.mark.parametrize("scale", [2.0 ** 110, 2.0 ** 100, 2.0 ** -100, 2.0 ** 60, 2.0 ** -60])
def test_xreg_extreme_activation_magnitudes(scale):
    M, N, K = 2, 40, 4096
    c = synth.q4_0_case(5300, N, K, M)
    x = (c["x"].astype(np.float64) * scale).astype(np.float32)
    y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(x), N=N)
    ref, bound = oracle.gemv_q4_0(c["w"], x, M, N, K)
    assert_parity(y, ref, bound, what=f"q4_0 x*{scale:g}")
    ck = synth.q4_k_case(5301, N, K, M)
    xk = (ck["x"].astype(np.float64) * scale).astype(np.float32)
    y = qg.qgemv_q4_k(to_dev(ck["w"]), to_dev(xk), N=N)
    ref, bound = oracle.gemv_q4_k(ck["w"], xk, M, N, K)
    assert_parity(y, ref, bound, what=f"q4_k x*{scale:g}")


def test_xreg_wide_activation_range_and_zeros():
    # One large element sets the power of two for the whole row; the rest
    # spans 2^-60 .. 2^10. Row 1 is all zeros (the result must be exactly 0).
    M, N, K = 2, 33, 4096
    c = synth.q4_0_case(5400, N, K, M)
    rng = np.random.default_rng(5)
    x = np.zeros((M, K), np.float32)
    x[0] = (rng.standard_normal(K) * 2.0 ** rng.integers(-60, 10, K)).astype(np.float32)
    x[0, 17] = 3.0e5
    y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(x), N=N)
    ref, bound = oracle.gemv_q4_0(c["w"], x, M, N, K)
    assert_parity(y, ref, bound, what="wide-range x")
    assert not y[1].any()


def test_xreg_non_finite_activation_propagates():
    M, N, K = 1, 20, 1024
    c = synth.q4_0_case(5500, N, K, M)
    for bad in (np.inf, np.nan):
        x = c["x"].copy()
        x[0, 100] = bad
        y = qg.qgemv_q4_0(to_dev(c["w"]), to_dev(x), N=N).cpu().numpy()
        assert not np.isfinite(y).any(), bad


@pytest.mark.parametrize("ahead", [1, 2, 5])
def test_xreg_ahead_does_not_change_results(ahead):
    M, N, K = 1, 700, 4096
    c = synth.q4_0_case(5600 + ahead, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    base = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    qg.set_option(qg.QG_OPT_XREG_AHEAD, ahead)
    try:
        ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    finally:
        qg.set_option(qg.QG_OPT_XREG_AHEAD, 0)
    assert_bitwise(ya, base[0], f"ahead={ahead} y_a")
    assert_bitwise(yb, base[1], f"ahead={ahead} y_b")


@pytest.mark.parametrize("M", [1, 2])
def test_xreg_agrees_with_staged_kernel(M):
    N, K = 257, 4096
    c = synth.q4_k_case(5700 + M, N, K, M)
    w, x = to_dev(c["w"]), to_dev(c["x"])
    y_new = qg.qgemv_q4_k(w, x, N=N)
    qg.set_option(qg.QG_OPT_XREG, 0)
    try:
        y_old = qg.qgemv_q4_k(w, x, N=N)
    finally:
        qg.set_option(qg.QG_OPT_XREG, 1)
    _, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
    # Both are within the bound of the exact value, so within twice of each other.
    assert_parity(y_new, y_old.cpu().numpy().astype(np.float64), bound, rel=2e-5, abs_=2e-6,
                  what="xreg vs staged")


def test_xreg_pdl_chain_at_full_size():
    """Back-to-back calls under programmatic dependent launch, each reading the
    previous call's output as its x (the decode-layer pattern)."""
    N = K = 4096
    c = synth.q4_0_case(5800, N, K, 1, dual=True)
    ck = synth.q4_k_case(5801, N, K, 1)
    wa, wb, wk = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(ck["w"])
    qg.set_option(qg.QG_OPT_PDL, 1)
    try:
        ya, yb = qg.qgemv_dual_q4_0(wa, wb, to_dev(c["x"]), N=N)
        y2 = qg.qgemv_q4_k(wk, yb, N=N)
        y3, y4 = qg.qgemv_dual_q4_0(wa, wb, y2, N=N)
        torch.cuda.synchronize()
    finally:
        qg.set_option(qg.QG_OPT_PDL, 0)
    _, (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], 1, N, K)
    assert_parity(yb, rb, bb, what="chain 1")
    r2, b2 = oracle.gemv_q4_k(ck["w"], yb.cpu().numpy(), 1, N, K)
    assert_parity(y2, r2, b2, what="chain 2")
    (r3, b3), _ = oracle.gemv_dual_q4_0(c["w"], c["w_b"], y2.cpu().numpy(), 1, N, K)
    assert_parity(y3, r3, b3, what="chain 3")
    assert qg.device_error() == 0


def test_xreg_independent_calls_mode():
    """QG_OPT_PDL = 2: consecutive calls that neither read nor write each
    other's buffers run concurrently; every output is bitwise what the same
    call gives alone."""
    N = K = 4096
    cases = [synth.q4_0_case(5900 + i, N, K, 1, dual=True) for i in range(3)]
    ws = [(to_dev(c["w"]), to_dev(c["w_b"])) for c in cases]
    x = to_dev(cases[0]["x"])
    alone = [qg.qgemv_dual_q4_0(wa, wb, x, N=N) for wa, wb in ws]
    torch.cuda.synchronize()
    outs = [(torch.empty((1, N), device="cuda"), torch.empty((1, N), device="cuda"))
            for _ in range(12)]
    qg.set_option(qg.QG_OPT_PDL, 2)
    try:
        for i, (ya, yb) in enumerate(outs):
            wa, wb = ws[i % 3]
            qg.qgemv_dual_q4_0(wa, wb, x, ya, yb, N=N)
        torch.cuda.synchronize()
    finally:
        qg.set_option(qg.QG_OPT_PDL, 0)
    for i, (ya, yb) in enumerate(outs):
        assert_bitwise(ya, alone[i % 3][0], f"independent call {i} y_a")
        assert_bitwise(yb, alone[i % 3][1], f"independent call {i} y_b")
    assert qg.device_error() == 0


@pytest.fixture(params=["automatic", "4 warps", "8 warps", "16 warps"])
def cta_shape(request):
    """The kernel's CTA shapes: automatic (eight consumer warps here, two CTAs
    per SM), four (four CTAs per SM, taken automatically for independent
    calls), eight, and sixteen (one CTA per SM). A count the shape does not
    allow falls back to automatic."""
    w = {"automatic": 0, "4 warps": 4, "8 warps": 8, "16 warps": 16}[request.param]
    qg.set_option(qg.QG_OPT_XREG_WARPS, w)
    yield request.param
    qg.set_option(qg.QG_OPT_XREG_WARPS, 0)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(37, 256), (61, 1024), (70, 3072), (300, 4096)])
def test_xreg_cta_shapes_q4_0(M, N, K, cta_shape):
    c = synth.q4_0_case(6000 + 7 * M + N, N, K, M, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    assert_bitwise(ya, qg.qgemv_q4_0(wa, x, N=N), f"{cta_shape} dual vs single")
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ya, ra, ba, what=f"{cta_shape} y_a M={M} N={N} K={K}")
    assert_parity(yb, rb, bb, what=f"{cta_shape} y_b M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2])
def test_xreg_cta_shapes_q4_k_and_affine(M, cta_shape):
    N, K = 129, 4096
    c = synth.q4_k_case(6100 + M, N, K, M)
    y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
    assert_parity(y, *oracle.gemv_q4_k(c["w"], c["x"], M, N, K), what=f"{cta_shape} q4_k")
    c = synth.affine_case(6200 + M, N, K, M, 64)
    x, s, b = to_dev(c["x"]), to_dev(c["s"]), to_dev(c["b"])
    yu = qg.qmm_affine(x, to_dev(c["q"]), s, b, 64, 0)
    yp = qg.qmm_affine(x, to_dev(c["q_packed"]), s, b, 64, 1)
    assert_bitwise(yp, yu, f"{cta_shape} packed vs u8")
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, 64, False)
    assert_parity(yu, ref, bound, what=f"{cta_shape} affine")


def test_xreg_cta_shape_does_not_change_results():
    """Each output's arithmetic depends on the format, M, K and x only: every
    CTA shape gives bitwise the same y."""
    N, K = 777, 4096
    c = synth.q4_0_case(6300, N, K, 1, dual=True)
    wa, wb, x = to_dev(c["w"]), to_dev(c["w_b"]), to_dev(c["x"])
    base = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    try:
        for warps in (4, 8, 16):
            qg.set_option(qg.QG_OPT_XREG_WARPS, warps)
            for ctas in (0, 1, 2, 4):
                qg.set_option(qg.QG_OPT_XREG_CTAS, ctas)
                ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
                assert_bitwise(ya, base[0], f"{warps} warps, {ctas} CTAs per SM, y_a")
                assert_bitwise(yb, base[1], f"{warps} warps, {ctas} CTAs per SM, y_b")
    finally:
        qg.set_option(qg.QG_OPT_XREG_WARPS, 0)
        qg.set_option(qg.QG_OPT_XREG_CTAS, 0)


@pytest.mark.parametrize("M", [3, 4, 5, 7, 8, 11])
@pytest.mark.parametrize("N,K", [(37, 256), (61, 1024), (130, 4096)])
def test_xreg_four_row_slices(M, N, K):
    """Three to eight (and more) rows of x run in slices of four rows on this
    kernel for Q4_K and affine weights with K <= 4096; a slice of three runs
    with one row of zeros. (Q4_0 keeps the staged kernel for M >= 3.)"""
    assert qg.workspace_size(qg.QG_OP_Q4_K, M, N, K) == 0
    ck = synth.q4_k_case(6500 + M + N, N, K, M)
    y = qg.qgemv_q4_k(to_dev(ck["w"]), to_dev(ck["x"]), N=N)
    assert_parity(y, *oracle.gemv_q4_k(ck["w"], ck["x"], M, N, K), what=f"q4_k M={M} K={K}")
    if K >= 256:
        ca = synth.affine_case(6600 + M + N, N, K, M, 64)
        xa, s_, b_ = to_dev(ca["x"]), to_dev(ca["s"]), to_dev(ca["b"])
        yu = qg.qmm_affine(xa, to_dev(ca["q"]), s_, b_, 64, 0)
        yp = qg.qmm_affine(xa, to_dev(ca["q_packed"]), s_, b_, 64, 1)
        assert_bitwise(yp, yu, f"M={M} packed vs u8")
        ref, bound = oracle.qmm_affine(ca["x"], ca["q"], ca["s"], ca["b"], M, N, K, 64, False)
        assert_parity(yu, ref, bound, what=f"affine M={M} K={K}")
    assert qg.device_error() == 0


def test_xreg_four_rows_full_size():
    """The decode sweep's M = 4 and 8 FFN-up Q4_K projection (N = 12288,
    K = 4096) and config 3's affine M = 8, sampled rows."""
    N, K = 12288, 4096
    for M in (4, 8):
        c = synth.q4_k_case(6700 + M, N, K, M)
        y = qg.qgemv_q4_k(to_dev(c["w"]), to_dev(c["x"]), N=N)
        rows = np.arange(3, N, 97)
        ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K, rows=rows)
        assert_parity(y.cpu().numpy()[:, rows], ref[:, rows], bound[:, rows], what=f"q4_k M={M}")
    c = synth.affine_case(6800, 4096, 4096, 8, 64)
    y = qg.qmm_affine(to_dev(c["x"]), to_dev(c["q"]), to_dev(c["s"]), to_dev(c["b"]), 64, 0)
    rows = np.arange(5, 4096, 61)
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], 8, 4096, 4096, 64, False,
                                   rows=rows)
    assert_parity(y.cpu().numpy()[:, rows], ref[:, rows], bound[:, rows], what="affine M=8")


def test_decode_layer_chain_under_pdl():
    """The decode layer's four full-size projections (Q+gate dual N = 4096,
    K+V dual N = 1024, FFN up Q4_K N = 12288, FFN down Q4_K K = 12288) in
    sequence under programmatic dependent launch, each reading the previous
    call's output as its x (chained where the shapes allow), against the
    oracle run on the same inputs."""
    H, F = 4096, 12288
    qgate = synth.q4_0_case(6900, H, H, 1, dual=True)
    kv = synth.q4_0_case(6901, H // 4, H, 1, dual=True)
    up = synth.q4_k_case(6902, F, H, 1)
    down = synth.q4_k_case(6903, H, F, 1)
    d = {k: to_dev(v) for k, v in (("qa", qgate["w"]), ("qb", qgate["w_b"]), ("ka", kv["w"]),
                                   ("kb", kv["w_b"]), ("up", up["w"]), ("down", down["w"]))}
    x0 = to_dev(qgate["x"])
    qg.set_option(qg.QG_OPT_PDL, 1)
    try:
        q, g = qg.qgemv_dual_q4_0(d["qa"], d["qb"], x0, N=H)     # x of K+V and FFN up: q
        k, v = qg.qgemv_dual_q4_0(d["ka"], d["kb"], q, N=H // 4)
        u = qg.qgemv_q4_k(d["up"], q, N=F)                         # FFN up reads q
        y = qg.qgemv_q4_k(d["down"], u, N=H)                       # FFN down reads u
        torch.cuda.synchronize()
    finally:
        qg.set_option(qg.QG_OPT_PDL, 0)
    (rq, bq), _ = oracle.gemv_dual_q4_0(qgate["w"], qgate["w_b"], qgate["x"], 1, H, H)
    assert_parity(q, rq, bq, what="Q+gate")
    qh = q.cpu().numpy()
    (rk, bk), (rv, bv) = oracle.gemv_dual_q4_0(kv["w"], kv["w_b"], qh, 1, H // 4, H)
    assert_parity(k, rk, bk, what="K")
    assert_parity(v, rv, bv, what="V")
    ru, bu = oracle.gemv_q4_k(up["w"], qh, 1, F, H)
    assert_parity(u, ru, bu, what="FFN up")
    ry, by = oracle.gemv_q4_k(down["w"], u.cpu().numpy(), 1, H, F)
    assert_parity(y, ry, by, what="FFN down")
    assert qg.device_error() == 0
