"""Pins for the oracle's quantizer round trips and GEMV references (CPU only).

* Round trips: weights that the format represents exactly must come back
  bit for bit through synth's encoder and the oracle's decoder, two pieces
  of code written separately.
* Closed forms: integer inputs give exact integer outputs, checked against
  numpy integer matrix products built from the codes themselves.
* Brute force: the f64 references equal numpy's f64 matmul of the
  dequantized weights (a library routine), and bound equals sum |x w|.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_gemv_dequant_gb300 import synth


# ----------------------------------------------------------------- round trips
def test_q4_0_roundtrip_representable_blocks():
    rng = np.random.default_rng(1)
    N, K = 16, 256
    nb = K // 32
    # d: positive fp16 values, so the code-0 element (-8d) is the unique
    # largest magnitude (codes stay below 16, so |q-8| <= 7 elsewhere).
    d16 = (rng.random((N, nb)) * 0.05 + 0.001).astype(np.float16)
    q = rng.integers(1, 16, size=(N, nb, 32)).astype(np.uint8)
    q[..., rng.integers(0, 32)] = 0
    W = ((q.astype(np.float32) - 8.0) * d16.astype(np.float32)[..., None]).reshape(N, K)
    enc = synth.quantize_q4_0(W)
    assert np.array_equal(enc, synth.q4_0_from_parts(d16.view(np.uint16), q))
    dec = oracle.dequant_q4_0(enc, N, K)
    assert np.array_equal(dec.view(np.uint32), W.view(np.uint32))


def test_q4_0_quantizer_error_bound():
    W = synth.normal(21, (64, 512), 0.02)
    enc = synth.quantize_q4_0(W)
    dec = oracle.dequant_q4_0(enc, 64, 512)
    d = np.abs(np.array([oracle.half_to_float(int(enc[n, 18 * b]) | (int(enc[n, 18 * b + 1]) << 8))
                         for n in range(64) for b in range(16)], dtype=np.float64)).reshape(64, 16)
    err = np.abs(dec.astype(np.float64) - W).reshape(64, 16, 32)
    # Half a step, except an element equal to -amax (w/d = +8) clamps to
    # q = 15, one full step; plus the fp16 rounding of d times |q-8| <= 8.
    lim_half = d[..., None] * (0.5 + 8 * 2.0 ** -10) + 1e-12
    lim_full = d[..., None] * (1.0 + 8 * 2.0 ** -10) + 1e-12
    assert np.all(err <= lim_full)
    assert np.mean(err <= lim_half) > 0.99


def test_q4_k_roundtrip_representable_superblocks():
    rng = np.random.default_rng(2)
    N, K = 8, 512
    nb = K // 256
    d16 = np.full((N, nb), 2.0 ** -9, dtype=np.float16) * (1 + rng.integers(0, 8, (N, nb))).astype(np.float16)
    dmin16 = np.full((N, nb), 2.0 ** -8, dtype=np.float16) * (1 + rng.integers(0, 8, (N, nb))).astype(np.float16)
    sc = np.full((N, nb, 8), 63, dtype=np.uint8)
    m = np.full((N, nb, 8), 63, dtype=np.uint8)
    q = rng.integers(0, 16, size=(N, nb, 8, 32)).astype(np.uint8)
    q[..., 0] = 0
    q[..., 1] = 15
    q = q.reshape(N, nb, 256)
    ref = synth.q4_k_from_parts(d16.view(np.uint16), dmin16.view(np.uint16), sc, m, q)
    W = oracle.dequant_q4_k(ref, N, K)
    enc = synth.quantize_q4_k(W)
    assert np.array_equal(enc, ref)


def test_q4_k_quantizer_error_bound():
    N, K = 32, 1024
    W = synth.normal(22, (N, K), 0.02)
    enc = synth.quantize_q4_k(W)
    dec = oracle.dequant_q4_k(enc, N, K).astype(np.float64)
    blk = enc.reshape(N, K // 256, 144)
    for n in range(0, N, 7):
        for b in range(K // 256):
            raw = blk[n, b]
            d = oracle.half_to_float(int(raw[0]) | (int(raw[1]) << 8))
            dmin = oracle.half_to_float(int(raw[2]) | (int(raw[3]) << 8))
            for j in range(8):
                sc, m = oracle.q4_k_scale_min(raw[4:16], j)
                sl = slice(256 * b + 32 * j, 256 * b + 32 * j + 32)
                step = d * sc
                # within half a step of the grid, plus clamp slack for the
                # rounded 6-bit scale/min (at most half a unit of d*15, dmin).
                lim = step / 2 + d * 15 / 2 + dmin / 2 + 1e-9
                assert np.max(np.abs(dec[n, sl] - W[n, sl])) <= lim


# ------------------------------------------------------------------ closed forms
def test_q4_0_integer_closed_form_exact():
    rng = np.random.default_rng(4)
    M, N, K = 3, 5, 256
    nb = K // 32
    q = rng.integers(0, 16, size=(N, nb, 32)).astype(np.uint8)
    w = synth.q4_0_from_parts(np.full((N, nb), 0x3C00, dtype=np.uint16), q)  # d = 1
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    ref, bound = oracle.gemv_q4_0(w, x, M, N, K)
    qi = q.reshape(N, K).astype(np.int64) - 8
    xi = x.astype(np.int64)
    assert np.array_equal(ref, (xi @ qi.T).astype(np.float64))
    assert np.array_equal(bound, (np.abs(xi) @ np.abs(qi).T).astype(np.float64))


def test_affine_unit_scale_is_dense_u8_gemv():
    rng = np.random.default_rng(5)
    M, N, K, gs = 2, 7, 128, 64
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    s = np.ones((N, K // gs), dtype=np.float32)
    b = np.zeros((N, K // gs), dtype=np.float32)
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    for packed in (False, True):
        qq = synth.pack_nibbles(q) if packed else q
        ref, _ = oracle.qmm_affine(x, qq, s, b, M, N, K, gs, packed)
        assert np.array_equal(ref, (x.astype(np.int64) @ q.astype(np.int64).T).astype(np.float64))


def test_q4_k_integer_closed_form_exact():
    rng = np.random.default_rng(6)
    M, N, K = 2, 4, 512
    nb = K // 256
    sc = rng.integers(0, 64, size=(N, nb, 8)).astype(np.uint8)
    m = rng.integers(0, 64, size=(N, nb, 8)).astype(np.uint8)
    q = rng.integers(0, 16, size=(N, nb, 256)).astype(np.uint8)
    w = synth.q4_k_from_parts(np.full((N, nb), 0x3C00, np.uint16), np.full((N, nb), 0x3C00, np.uint16),
                              sc, m, q)  # d = dmin = 1
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    ref, _ = oracle.gemv_q4_k(w, x, M, N, K)
    sub = np.arange(K) % 256 // 32
    wi = (sc[:, np.arange(K) // 256, sub].astype(np.int64) * q.reshape(N, K).astype(np.int64)
          - m[:, np.arange(K) // 256, sub].astype(np.int64))
    assert np.array_equal(ref, (x.astype(np.int64) @ wi.T).astype(np.float64))


# ------------------------------------------------------------------ brute force
@pytest.mark.parametrize("M,N,K", [(1, 5, 32), (3, 4, 64), (2, 3, 512)])
def test_q4_0_gemv_vs_numpy_matmul(M, N, K):
    case = synth.q4_0_case(30 + K, N, K, M)
    W = oracle.dequant_q4_0(case["w"], N, K).astype(np.float64)
    x = case["x"].astype(np.float64)
    ref, bound = oracle.gemv_q4_0(case["w"], case["x"], M, N, K)
    np.testing.assert_allclose(ref, x @ W.T, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(bound, np.abs(x) @ np.abs(W).T, rtol=1e-12, atol=1e-15)
    assert np.all(bound >= np.abs(ref))


@pytest.mark.parametrize("M,N,K", [(1, 3, 256), (3, 5, 512)])
def test_q4_k_gemv_vs_numpy_matmul(M, N, K):
    case = synth.q4_k_case(40 + K, N, K, M)
    W = oracle.dequant_q4_k(case["w"], N, K).astype(np.float64)
    ref, bound = oracle.gemv_q4_k(case["w"], case["x"], M, N, K)
    x = case["x"].astype(np.float64)
    np.testing.assert_allclose(ref, x @ W.T, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(bound, np.abs(x) @ np.abs(W).T, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("packed", [False, True])
def test_affine_qmm_vs_numpy_matmul(packed):
    M, N, K, gs = 3, 6, 256, 64
    case = synth.affine_case(50, N, K, M, gs)
    qq = case["q_packed"] if packed else case["q"]
    W = oracle.dequant_affine(qq, case["s"], case["b"], N, K, gs, packed).astype(np.float64)
    ref, bound = oracle.qmm_affine(case["x"], qq, case["s"], case["b"], M, N, K, gs, packed)
    x = case["x"].astype(np.float64)
    np.testing.assert_allclose(ref, x @ W.T, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(bound, np.abs(x) @ np.abs(W).T, rtol=1e-12, atol=1e-15)


def test_row_subset_matches_full():
    M, N, K = 2, 9, 128
    case = synth.q4_0_case(60, N, K, M)
    full, fb = oracle.gemv_q4_0(case["w"], case["x"], M, N, K)
    rows = [8, 0, 3]
    part, pb = oracle.gemv_q4_0(case["w"], case["x"], M, N, K, rows=rows)
    assert np.array_equal(part[:, rows], full[:, rows])
    assert np.array_equal(pb[:, rows], fb[:, rows])


def test_dual_equals_two_singles():
    M, N, K = 2, 6, 128
    case = synth.q4_0_case(61, N, K, M, dual=True)
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(case["w"], case["w_b"], case["x"], M, N, K)
    sa, sba = oracle.gemv_q4_0(case["w"], case["x"], M, N, K)
    sb, sbb = oracle.gemv_q4_0(case["w_b"], case["x"], M, N, K)
    assert np.array_equal(ra, sa) and np.array_equal(rb, sb)
    assert np.array_equal(ba, sba) and np.array_equal(bb, sbb)


def test_tolerance_helper():
    ref = np.array([1.0, -2.0])
    bound = np.array([10.0, 10.0])
    ok, ratio = oracle.within(np.array([1.0 + 5e-5, -2.0 - 2e-4]), ref, bound)
    assert ok.tolist() == [True, False] and ratio > 1
