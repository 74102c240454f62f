"""GPU parity for the tensor-core affine prefill path of qmm_affine.

Tolerance (per output, the bar for the tensor-core path):
    |y - ref| <= 2e-3 * sum_k |x_k w_k| + 1e-6
with ref and the sum from the oracle in f64. A second, tighter check pins the
path's one approximation: rounding each activation row, scaled by a power of
two, to fp16. Feeding those rounded activations to the oracle must reproduce
y within the f32 bar (1e-5), so no other error source (a wrong group, scale,
bias or tile) can hide inside the looser tolerance. The folded-weight kernel
(QG_OPT_PREFILL_FOLD = 1) also rounds each weight row, scaled by a power of
two, to fp16; its tighter check feeds the oracle both rounded operands. Every
tensor-core test runs on both kernels.

Shapes span several 128x128 tiles with ragged tails in M, N and K, every
group size the path takes (16 .. 1024), both code storages, 8-bit codes, and
the full 512 x 4096 x 4096 workload that the benchmark times.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, dev, to_dev

pytestmark = pytest.mark.gpu

REL_TC = oracle.REL_TC


@pytest.fixture(autouse=True)
def tensor_cores_from_m16():
    """These tests exercise the tensor-core prefill at small M on purpose: the
    threshold is lowered to 16 for them (the library's default is 64)."""
    old = qg.get_option(qg.QG_OPT_PREFILL_MIN_M)
    qg.set_option(qg.QG_OPT_PREFILL_MIN_M, 16)
    yield
    qg.set_option(qg.QG_OPT_PREFILL_MIN_M, old)


@pytest.fixture
def min_m():
    old = qg.get_option(qg.QG_OPT_PREFILL_MIN_M)
    yield
    qg.set_option(qg.QG_OPT_PREFILL_MIN_M, old)


@pytest.fixture(params=["exact", "fold"])
def kernel(request):
    """Selects the prefill kernel; the value is true for the exact-code one."""
    old = qg.get_option(qg.QG_OPT_PREFILL_FOLD)
    qg.set_option(qg.QG_OPT_PREFILL_FOLD, int(request.param == "fold"))
    yield request.param == "exact"
    qg.set_option(qg.QG_OPT_PREFILL_FOLD, old)


def _run(c, gs, packed, M=None):
    q = c["q_packed"] if packed else c["q"]
    return qg.qmm_affine(to_dev(c["x"]), to_dev(q), to_dev(c["s"]), to_dev(c["b"]), gs, packed)


def _rounded_x(x):
    """x scaled per row by 2^e (largest |x| into [2^14, 2^15)), rounded to fp16
    and scaled back: the activations the tensor-core path multiplies."""
    x = np.asarray(x, dtype=np.float32)
    out = np.empty_like(x)
    for m in range(x.shape[0]):
        amax = float(np.max(np.abs(x[m]))) if x.shape[1] else 0.0
        e = 0
        if 0.0 < amax < np.inf:
            _, ex = np.frexp(np.float32(amax))
            e = int(min(126, max(-126, 15 - int(ex))))
        sc = np.float32(np.ldexp(np.float32(1.0), e))
        h = (x[m] * sc).astype(np.float16).astype(np.float32)
        out[m] = h * np.float32(np.ldexp(np.float32(1.0), -e))
    return out


def _rounded_w(W, rowbound):
    """The folded kernel's weights: row n scaled by 2^f (f puts the row's bound
    max_g (|s| qmax + |b|) into [2^14, 2^15)), rounded to fp16, scaled back."""
    W = np.asarray(W, dtype=np.float64)
    out = np.empty(W.shape, dtype=np.float32)
    for n in range(W.shape[0]):
        bm = np.float32(rowbound[n])
        f = 0
        if 0.0 < bm < np.inf:
            _, ex = np.frexp(bm)
            f = int(min(120, max(-120, 15 - int(ex))))
        h = np.ldexp(W[n], f).astype(np.float16).astype(np.float64)
        out[n] = np.ldexp(h, -f).astype(np.float32)
    return out


def affine_rowbound(s, b, qmax):
    return np.max(np.abs(np.asarray(s, np.float32)) * np.float32(qmax)
                  + np.abs(np.asarray(b, np.float32)), axis=1)


def rounded_ref(x, W, rowbound, M, N, K):
    """Oracle (f64) on the operands the folded kernel multiplies."""
    return oracle.gemv_dense(_rounded_w(W, rowbound), _rounded_x(x), M, N, K)


def check_rounding_only(y, kernel, x, q, s, b, M, N, K, gs, qmax, what):
    """The f32 bar against the oracle fed the kernel's rounded operands."""
    if kernel:
        ref, bound = oracle.qmm_affine(_rounded_x(x), q, s, b, M, N, K, gs, False)
    else:
        W = oracle.dequant_affine(q, s, b, N, K, gs, False)
        ref, bound = rounded_ref(x, W, affine_rowbound(s, b, qmax), M, N, K)
    assert_parity(y, ref, bound, what=what)


SHAPES = [
    # M,   N,   K,    gs
    (16, 128, 256, 64),
    (130, 200, 512, 32),
    (257, 385, 320, 64),
    (128, 128, 1024, 128),
    (40, 96, 2048, 256),
    (33, 70, 2048, 1024),
    (64, 136, 128, 16),
    (20, 150, 96, 32),     # K not a multiple of the 64-wide stage
    (24, 130, 64, 32),     # a single stage
    (40, 64, 32, 16),      # a single, partial stage
]


@pytest.mark.parametrize("M,N,K,gs", SHAPES)
def test_prefill_parity_and_packed_equals_u8(M, N, K, gs, kernel):
    c = synth.affine_case(4100 + M + N + gs, N, K, M, gs)
    yu = _run(c, gs, 0)
    yp = _run(c, gs, 1)
    assert_bitwise(yp, yu, f"prefill packed vs u8 M={M} N={N} K={K} gs={gs}")
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(yu, ref, bound, rel=REL_TC, what=f"prefill M={M} N={N} K={K} gs={gs}")


@pytest.mark.parametrize("M,N,K,gs", SHAPES[:4])
def test_prefill_error_is_only_fp16_rounding(M, N, K, gs, kernel):
    c = synth.affine_case(4200 + M + gs, N, K, M, gs)
    y = _run(c, gs, 0)
    check_rounding_only(y, kernel, c["x"], c["q"], c["s"], c["b"], M, N, K, gs, 255,
                        f"prefill vs rounded-operand oracle M={M} gs={gs}")
    yp = _run(c, gs, 1)
    check_rounding_only(yp, kernel, c["x"], c["q"], c["s"], c["b"], M, N, K, gs, 15,
                        f"packed prefill vs rounded-operand oracle M={M} gs={gs}")


def test_prefill_8bit_codes(kernel):
    M, N, K, gs = 200, 300, 1024, 64
    c = synth.affine_case(4300, N, K, M, gs)
    q8 = synth.codes(4301, (N, K), bits=8)
    y = qg.qmm_affine(to_dev(c["x"]), to_dev(q8), to_dev(c["s"]), to_dev(c["b"]), gs, 0)
    ref, bound = oracle.qmm_affine(c["x"], q8, c["s"], c["b"], M, N, K, gs, False)
    assert_parity(y, ref, bound, rel=REL_TC, what="prefill 8-bit codes")
    check_rounding_only(y, kernel, c["x"], q8, c["s"], c["b"], M, N, K, gs, 255,
                        "prefill 8-bit codes vs rounded-operand oracle")


def test_prefill_row_scaling_extremes(kernel):
    """Rows far outside fp16's range (1e6, 1e-20) and an all-zero row: the
    per-row power-of-two scale keeps them exact up to fp16 rounding."""
    M, N, K, gs = 32, 160, 512, 64
    c = synth.affine_case(4400, N, K, M, gs)
    x = c["x"].copy()
    x[0] *= np.float32(1e6)
    x[1] *= np.float32(1e-20)
    x[2] = 0.0
    x[3, 5] = np.float32(3e4)  # one large element dominates the row's scale
    y = qg.qmm_affine(to_dev(x), to_dev(c["q"]), to_dev(c["s"]), to_dev(c["b"]), gs, 0)
    ref, bound = oracle.qmm_affine(x, c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(y, ref, bound, rel=REL_TC, what="prefill extreme rows")
    assert np.all(y.cpu().numpy()[2] == 0.0)


def test_prefill_weight_row_extremes(kernel):
    """Weight rows far outside fp16's range (scales and biases times 1e6 and
    1e-20), an all-zero row, and a row whose groups differ by 2^10 in scale:
    the folded kernel's per-row power of two keeps them within the bar."""
    M, N, K, gs = 40, 140, 512, 64
    c = synth.affine_case(4450, N, K, M, gs)
    s, b = c["s"].copy(), c["b"].copy()
    s[0] *= np.float32(1e6)
    b[0] *= np.float32(1e6)
    s[1] *= np.float32(1e-20)
    b[1] *= np.float32(1e-20)
    s[2] = 0.0
    b[2] = 0.0
    s[3, 1] *= np.float32(1024.0)
    b[3, 1] *= np.float32(1024.0)
    for packed in (0, 1):
        q = c["q_packed"] if packed else c["q"]
        y = qg.qmm_affine(to_dev(c["x"]), to_dev(q), to_dev(s), to_dev(b), gs, packed)
        ref, bound = oracle.qmm_affine(c["x"], c["q"], s, b, M, N, K, gs, False)
        assert_parity(y, ref, bound, rel=REL_TC, what=f"prefill extreme weight rows packed={packed}")
        check_rounding_only(y, kernel, c["x"], c["q"], s, b, M, N, K, gs, 15 if packed else 255,
                            f"extreme weight rows vs rounded-operand oracle packed={packed}")
        assert np.all(y.cpu().numpy()[:, 2] == 0.0)


@pytest.mark.parametrize("packed", [0, 1])
def test_prefill_full_workload_sampled(packed, kernel):
    """512 x 4096 x 4096, gs 64: the benchmarked launch. The oracle computes
    every activation row for 96 sampled weight rows, spread over all 32
    weight tiles (first and last row of each included)."""
    M, N, K, gs = 512, 4096, 4096, 64
    c = synth.affine_case(3, N, K, M, gs)
    x, s, b = to_dev(c["x"]), to_dev(c["s"]), to_dev(c["b"])
    yu = qg.qmm_affine(x, to_dev(c["q"]), s, b, gs, 0)
    if packed:
        yp = qg.qmm_affine(x, to_dev(c["q_packed"]), s, b, gs, 1)
        assert_bitwise(yp, yu, "full workload packed vs u8")
        return
    rows = np.unique(np.concatenate([np.arange(0, N, 128), np.arange(127, N, 128),
                                     np.random.default_rng(7).integers(0, N, 32)]))
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False, rows=rows)
    yh = yu.cpu().numpy()
    assert_parity(yh[:, rows], ref[:, rows], bound[:, rows], rel=REL_TC, what="full workload")


def test_prefill_min_m_option_selects_path(min_m, kernel):
    M, N, K, gs = 24, 96, 512, 64
    c = synth.affine_case(4500, N, K, M, gs)
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    qg.set_option(qg.QG_OPT_PREFILL_MIN_M, 1 << 20)  # CUDA cores: the f32 bar
    y_cc = _run(c, gs, 0)
    assert_parity(y_cc, ref, bound, what="CUDA-core path M=24")
    qg.set_option(qg.QG_OPT_PREFILL_MIN_M, 1)        # tensor cores, even M=1
    y_tc = _run(c, gs, 0)
    assert_parity(y_tc, ref, bound, rel=REL_TC, what="tensor-core path M=24")
    check_rounding_only(y_tc, kernel, c["x"], c["q"], c["s"], c["b"], M, N, K, gs, 255,
                        "tensor-core path M=24 vs rounded operands")
    c1 = synth.affine_case(4501, N, K, 1, gs)
    y1 = _run(c1, gs, 1)
    ref1, bound1 = oracle.qmm_affine(c1["x"], c1["q"], c1["s"], c1["b"], 1, N, K, gs, False)
    assert_parity(y1, ref1, bound1, rel=REL_TC, what="tensor-core path M=1")


def test_prefill_unaligned_codes_fall_back_to_cuda_cores():
    M, N, K, gs = 48, 64, 256, 64
    c = synth.affine_case(4600, N, K, M, gs)
    q = to_dev(c["q"], 1)  # codes one byte past a 16-byte boundary
    y = qg.qmm_affine(to_dev(c["x"]), q, to_dev(c["s"]), to_dev(c["b"]), gs, 0)
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(y, ref, bound, what="unaligned codes, CUDA-core bar")


def test_prefill_small_group_size_falls_back_to_cuda_cores():
    M, N, K, gs = 40, 50, 256, 8
    c = synth.affine_case(4700, N, K, M, gs)
    y = _run(c, gs, 0)
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(y, ref, bound, what="gs=8, CUDA-core bar")


def test_prefill_requires_workspace(kernel):
    M, N, K, gs = 64, 128, 256, 64
    need = qg.workspace_size(qg.QG_OP_AFFINE, M, N, K, gs, 0)
    assert need >= M * K * 2  # at least the fp16 copy of x
    c = synth.affine_case(4800, N, K, M, gs)
    x, q, s, b = to_dev(c["x"]), to_dev(c["q"]), to_dev(c["s"]), to_dev(c["b"])
    y = torch.empty((M, N), device=dev())
    ws = torch.empty(need // 4, dtype=torch.float32, device=dev())
    L = qg.lib()
    st = torch.cuda.current_stream().cuda_stream
    args = (x.data_ptr(), q.data_ptr(), s.data_ptr(), b.data_ptr(), y.data_ptr(), M, N, K, gs, 0)
    assert L.qmm_affine(*args, None, 0, st) == qg.QG_ERR_WORKSPACE
    assert L.qmm_affine(*args, C.c_void_p(ws.data_ptr()), need - 16, st) == qg.QG_ERR_WORKSPACE
    assert L.qmm_affine(*args, C.c_void_p(ws.data_ptr()), need, st) == qg.QG_OK
    ref, bound = oracle.qmm_affine(c["x"], c["q"], c["s"], c["b"], M, N, K, gs, False)
    assert_parity(y, ref, bound, rel=REL_TC, what="explicit workspace")


def test_prefill_no_device_error():
    assert qg.device_error() == 0
