"""GPU parity for the prepared AF4-g64 layout: qg_prepare_af4_g64 and
qmm_af4_g64 (qmm_affine.rs, mlx-native 0.21.1: prepare_af4_g64 and
dispatch_qmm_affine_t_packed_simd4_b4_gs64_bf16; M <= 32, N and K multiples
of 64, bf16 scale and bias per 64-group).

The prepared words must equal the oracle's bit for bit. qmm_af4_g64 is held to
the oracle's qmm_affine on the unprepared codes with the bf16 scales and
biases taken exactly as f32, under the f32 bar (1e-5 * sum |x w| + 1e-6) for
every M. Shapes cover one and two row blocks per CTA (odd and even N / 64),
one and several K slices per row block (a cluster of 1 to 8 CTAs), x staged
in more than one sub-slice (M = 32, K = 12288), odd group counts, every M
tile (8, 4, 2, 1) and the 4096 x 4096 workload the benchmark times; for M <= 2 and
K <= 4096 the register-resident-x kernel (agreement with the cluster kernel,
every launch mode, metadata off a 16-byte boundary falling back). Row m of y
must not depend on M within M in 1..2, 3..8 and 9..32, and x at a 4-byte
offset (the scalar staging path) must give bitwise the same y.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, dev, to_dev

pytestmark = pytest.mark.gpu


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(
        torch.bfloat16)


def _prepare(c):
    return qg.prepare_af4_g64(to_dev(c["q"]), _bf16(c["s_bits"]), _bf16(c["b_bits"]))


@pytest.mark.parametrize("N,K", [(64, 64), (192, 512), (128, 4096), (320, 128)])
def test_prepare_equals_oracle_bitwise(N, K):
    c = synth.af4_case(7000 + N + K, N, K, 1)
    plane, meta = _prepare(c)
    rp, rm = oracle.prepare_af4_g64(c["q"], c["s_bits"], c["b_bits"], N, K)
    assert_bitwise(plane.cpu().numpy(), rp.view(np.int32), f"af4 plane N={N} K={K}")
    assert_bitwise(meta.cpu().numpy(), rm.view(np.int32), f"af4 metadata N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2, 3, 8, 17, 31, 32])
@pytest.mark.parametrize("N,K", [(64, 64), (192, 512), (128, 1088), (64, 12288),
                                 (128, 12288)])
def test_qmm_af4_parity(M, N, K):
    c = synth.af4_case(7100 + M + N + K, N, K, M)
    plane, meta = _prepare(c)
    ref, bound = oracle.qmm_af4_g64(c["x"], c["q"], c["s_bits"], c["b_bits"], M, N, K)
    y = qg.qmm_af4_g64(to_dev(c["x"]), plane, meta, N)
    assert_parity(y, ref, bound, what=f"qmm_af4_g64 M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(192, 512), (64, 12288), (512, 4096)])
def test_qmm_af4_rows_do_not_depend_on_m(N, K):
    """Within each class of M (1..2 on the register-resident-x kernel when it
    takes the shape, 3..8 and 9..32 with one K slicing each) row m of y is
    bitwise the same whatever M is."""
    c = synth.af4_case(7200 + N, N, K, 32)
    plane, meta = _prepare(c)
    x = to_dev(c["x"])
    y32 = qg.qmm_af4_g64(x, plane, meta, N)
    for M in (9, 13, 31):
        yM = qg.qmm_af4_g64(x[32 - M:].contiguous(), plane, meta, N)
        assert_bitwise(yM, y32[32 - M:], f"af4 rows of M={M} vs M=32")
    y8 = qg.qmm_af4_g64(x[:8].contiguous(), plane, meta, N)
    for M in (3, 5):
        yM = qg.qmm_af4_g64(x[8 - M:8].contiguous(), plane, meta, N)
        assert_bitwise(yM, y8[8 - M:], f"af4 rows of M={M} vs M=8")
    y2 = qg.qmm_af4_g64(x[:2].contiguous(), plane, meta, N)
    y1 = qg.qmm_af4_g64(x[1:2].contiguous(), plane, meta, N)
    assert_bitwise(y1, y2[1:], "af4 rows of M=1 vs M=2")


def test_qmm_af4_unaligned_x_is_bitwise_equal():
    M, N, K = 9, 192, 512
    c = synth.af4_case(7250, N, K, M)
    plane, meta = _prepare(c)
    flat = torch.zeros(M * K + 1, dtype=torch.float32, device=dev())
    flat[1:] = torch.from_numpy(c["x"].ravel()).to(dev())
    xu = flat[1:].view(M, K)
    assert xu.data_ptr() % 16 == 4
    ya = qg.qmm_af4_g64(to_dev(c["x"]), plane, meta, N)
    yu = qg.qmm_af4_g64(xu, plane, meta, N)
    assert_bitwise(yu, ya, "af4 x at a 4-byte offset")


def test_qmm_af4_page_test_inputs():
    """The inputs of the page's own bounded-error test (m = 31, n = 64,
    k = 128: x = 0.5 sin(0.013 i - 0.7), code = (11 i + 3) mod 16, scale
    bf16(0.01 + 1e-4 i), bias bf16(-0.1 + 2e-4 i)) and its two bounds
    (relative RMSE and the largest error over max(|y|, 1), each at most
    5e-3), besides the tensor-core bar."""
    m, n, k = 31, 64, 128
    x = (np.sin(np.arange(m * k, dtype=np.float32) * np.float32(0.013) - np.float32(0.7))
         * np.float32(0.5)).astype(np.float32).reshape(m, k)
    q = ((np.arange(n * k) * 11 + 3) % 16).astype(np.uint8).reshape(n, k)
    i = np.arange(n * k // 64, dtype=np.float32)
    sb = synth.bf16_bits(np.float32(0.01) + i * np.float32(0.0001)).reshape(n, k // 64)
    bb = synth.bf16_bits(np.float32(-0.1) + i * np.float32(0.0002)).reshape(n, k // 64)
    plane, meta = qg.prepare_af4_g64(to_dev(q), _bf16(sb), _bf16(bb))
    y = qg.qmm_af4_g64(to_dev(x), plane, meta, n).cpu().numpy().astype(np.float64)
    ref, bound = oracle.qmm_af4_g64(x, q, sb, bb, m, n, k)
    assert_parity(y, ref, bound, what="qmm_af4_g64 page inputs")
    err = y - ref
    assert np.sqrt(np.sum(err * err) / np.sum(ref * ref)) <= 5e-3
    assert np.max(np.abs(err) / np.maximum(np.abs(ref), 1.0)) <= 5e-3


@pytest.mark.parametrize("M", [8, 32])
def test_qmm_af4_full_size_sampled(M):
    """The 4096 x 4096 workload the benchmark times, on sampled outputs."""
    N = K = 4096
    c = synth.af4_case(7300 + M, N, K, M)
    plane, meta = _prepare(c)
    y = qg.qmm_af4_g64(to_dev(c["x"]), plane, meta, N).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, N, 512), np.arange(63, N, 512),
                                     np.random.default_rng(M).integers(0, N, 32)]))
    ref, bound = oracle.qmm_af4_g64(c["x"], c["q"], c["s_bits"], c["b_bits"], M, N, K,
                                    rows=rows)
    assert_parity(y[:, rows], ref[:, rows], bound[:, rows], what=f"qmm_af4_g64 4096 M={M}")


def test_qmm_af4_validation():
    N, K = 64, 128
    c = synth.af4_case(7400, N, K, 33)
    plane, meta = _prepare(c)
    x = to_dev(c["x"])
    with pytest.raises(qg.QGError):
        qg.qmm_af4_g64(x, plane, meta, N)                   # M = 33 > 32
    with pytest.raises(qg.QGError):
        qg.qmm_af4_g64(x[:4, :96].contiguous(), plane, meta, N)   # K % 64 != 0
    with pytest.raises(qg.QGError):
        qg.qmm_af4_g64(x[:4], plane, meta, 96)              # N % 64 != 0
    assert qg.workspace_size(qg.QG_OP_AF4_G64, 4, N, K) == 0
    with pytest.raises(qg.QGError):                          # y overlaps x
        qg.qmm_af4_g64(x[:4], plane, meta, N, y=x[:4].reshape(-1)[:4 * N].view(4, N))
    with pytest.raises(qg.QGError):
        qg.prepare_af4_g64(to_dev(c["q"][:, :96].copy()), _bf16(c["s_bits"][:, :1].copy()),
                           _bf16(c["b_bits"][:, :1].copy()))   # K % 64 != 0


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(192, 512), (128, 1088), (256, 4096), (64, 64)])
def test_qmm_af4_register_path_agrees_with_cluster_kernel(M, N, K):
    """With one or two rows of x (K <= 4096, 16-byte aligned buffers) the
    register-resident-x kernel takes the call; with QG_OPT_XREG = 0 the
    cluster kernel does. Both are within the bound of the exact value, so
    within twice of each other."""
    c = synth.af4_case(7500 + M + N + K, N, K, M)
    plane, meta = _prepare(c)
    x = to_dev(c["x"])
    y_new = qg.qmm_af4_g64(x, plane, meta, N)
    qg.set_option(qg.QG_OPT_XREG, 0)
    try:
        y_old = qg.qmm_af4_g64(x, plane, meta, N)
    finally:
        qg.set_option(qg.QG_OPT_XREG, 1)
    ref, bound = oracle.qmm_af4_g64(c["x"], c["q"], c["s_bits"], c["b_bits"], M, N, K)
    assert_parity(y_new, ref, bound, what=f"af4 register path M={M} N={N} K={K}")
    assert_parity(y_new, y_old.cpu().numpy().astype(np.float64), bound, rel=2e-5, abs_=2e-6,
                  what=f"af4 register path vs cluster kernel M={M}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_qmm_af4_launch_modes(mode):
    """Every QG_OPT_PDL mode (launch shapes differ): outputs bitwise equal to
    the default mode's, and a chain whose x is the previous call's y."""
    N = K = 4096
    c = synth.af4_case(7600, N, K, 2)
    plane, meta = _prepare(c)
    x = to_dev(c["x"])
    base = qg.qmm_af4_g64(x, plane, meta, N)
    old = qg.get_option(qg.QG_OPT_PDL)
    qg.set_option(qg.QG_OPT_PDL, mode)
    try:
        y1 = qg.qmm_af4_g64(x, plane, meta, N)
        y2 = qg.qmm_af4_g64(y1, plane, meta, N) if mode != 2 else None
        torch.cuda.synchronize()
    finally:
        qg.set_option(qg.QG_OPT_PDL, old)
    assert_bitwise(y1, base, f"PDL mode {mode}")
    if y2 is not None:
        ref, bound = oracle.qmm_af4_g64(y1.cpu().numpy(), c["q"], c["s_bits"], c["b_bits"], 2,
                                        N, K)
        assert_parity(y2, ref, bound, what=f"chain under PDL mode {mode}")
    assert qg.device_error() == 0


def test_qmm_af4_metadata_off_16_bytes():
    """Metadata 4 bytes off a 16-byte boundary (allowed) keeps the call on the
    cluster kernel; results stay within the bar."""
    M, N, K = 2, 128, 1024
    c = synth.af4_case(7700, N, K, M)
    plane, meta = _prepare(c)
    buf = torch.zeros(meta.numel() + 4, dtype=torch.int32, device=dev())
    buf[1:1 + meta.numel()] = meta
    meta_u = buf[1:1 + meta.numel()]
    assert meta_u.data_ptr() % 16 == 4
    y = qg.qmm_af4_g64(to_dev(c["x"]), plane, meta_u, N)
    ref, bound = oracle.qmm_af4_g64(c["x"], c["q"], c["s_bits"], c["b_bits"], M, N, K)
    assert_parity(y, ref, bound, what="af4 metadata at a 4-byte offset")
