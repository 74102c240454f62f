"""Pins for the oracle's format decoders (CPU only).

Each test checks the oracle against something other than itself: numpy's
IEEE half conversion, blocks decoded by hand (tests/golden), the page's u32
packing rule, or an exact algebraic identity.
"""
import json
import os

import numpy as np
import pytest

import oracle
from bit_quantized_gemv_dequant_gb300 import synth

from conftest import GOLDEN


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_half_decoder_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_float_array(bits)
    theirs = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), theirs[~nan].view(np.uint32))


@pytest.mark.parametrize("bits,val", [(0x3C00, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -24),
                                      (0x7BFF, 65504.0), (0x0400, 2.0 ** -14), (0x8000, -0.0),
                                      (0x3555, 1365.0 / 4096.0)])
def test_half_decoder_hand_values(bits, val):
    got = oracle.half_to_float(bits)
    assert np.float32(got).view(np.uint32) == np.float32(val).view(np.uint32)


def test_q4_0_golden_blocks():
    fx = _load("q4_0_blocks.json")
    for blk in fx["blocks"]:
        raw = np.frombuffer(bytes.fromhex(blk["hex"]), dtype=np.uint8)
        got = oracle.q4_0_block(raw)
        exp = np.array(blk["expected"], dtype=np.float32)
        assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), blk["name"]


def test_q4_0_dequant_matrix_matches_blocks():
    fx = _load("q4_0_blocks.json")
    raw = np.concatenate([np.frombuffer(bytes.fromhex(b["hex"]), dtype=np.uint8)
                          for b in fx["blocks"][:4]])
    got = oracle.dequant_q4_0(raw, 2, 64)
    exp = np.array(sum((b["expected"] for b in fx["blocks"][:4]), []), dtype=np.float32)
    assert np.array_equal(got.ravel().view(np.uint32), exp.view(np.uint32))


def _q4_k_golden_block(sb, rule_j_l):
    header = np.frombuffer(bytes.fromhex(sb["header_hex"]), dtype=np.uint8)
    q = np.array([[rule_j_l(j, l) for l in range(32)] for j in range(8)], dtype=np.uint8)
    qs = np.empty(128, dtype=np.uint8)
    for c in range(4):
        qs[32 * c:32 * c + 32] = q[2 * c] | (q[2 * c + 1] << 4)
    return np.concatenate([header, qs]), q


def test_q4_k_golden_superblocks():
    fx = _load("q4_k_superblocks.json")
    rule = lambda j, l: (l + 3 * j) % 16
    for sb in fx["superblocks"]:
        raw, q = _q4_k_golden_block(sb, rule)
        for j in range(8):
            assert oracle.q4_k_scale_min(raw[4:16], j) == (sb["sc"][j], sb["m"][j]), (sb["name"], j)
        got = oracle.q4_k_block(raw)
        for j in range(8):
            for l in range(32):
                exp = sb["d"] * sb["sc"][j] * int(q[j, l]) - sb["dmin"] * sb["m"][j]
                # Both products are exact dyadic values here, so exp is exact.
                assert got[32 * j + l] == np.float32(exp), (sb["name"], j, l)


def test_q4_k_scale_packing_roundtrip_all_pairs():
    # Every 6-bit value in every sub-block slot survives pack -> oracle unpack.
    rng = np.random.default_rng(7)
    for _ in range(200):
        sc = rng.integers(0, 64, size=8)
        m = rng.integers(0, 64, size=8)
        s12 = synth.pack_q4_k_scales(sc, m)
        for j in range(8):
            assert oracle.q4_k_scale_min(s12, j) == (sc[j], m[j])


def test_affine_pack_matches_u32_word_rule():
    fx = _load("affine_pack.json")
    for item in fx["words"]:
        word = int(item["word"], 16)
        codes = np.array(item["codes"], dtype=np.uint8)[None, :]
        packed = synth.pack_nibbles(codes)
        assert bytes(packed.ravel()) == word.to_bytes(4, "little")


def test_affine_golden_dequant():
    fx = _load("affine_pack.json")
    for item in fx["dequant"]:
        q = np.array([[item["q"], 0]], dtype=np.uint8)
        s = np.array([[item["s"]]], dtype=np.float32)
        b = np.array([[item["b"]]], dtype=np.float32)
        got = oracle.dequant_affine(q, s, b, 1, 2, 2, False)
        assert got[0, 0] == np.float32(item["w"])


def test_affine_packed_equals_u8_bitwise():
    case = synth.affine_case(11, 24, 256, 1, 64)
    a = oracle.dequant_affine(case["q"], case["s"], case["b"], 24, 256, 64, False)
    p = oracle.dequant_affine(case["q_packed"], case["s"], case["b"], 24, 256, 64, True)
    assert np.array_equal(a.view(np.uint32), p.view(np.uint32))


def test_affine_single_rounding():
    # fmaf(q, s, b) rounds once: pick values where q*s rounds differently
    # from q*s+b computed exactly, and compare with the f64 value rounded once.
    rng = np.random.default_rng(3)
    q = rng.integers(0, 16, size=(8, 128)).astype(np.uint8)
    s = rng.random((8, 2), dtype=np.float32) * np.float32(0.01) + np.float32(0.001)
    b = -rng.random((8, 2), dtype=np.float32) * np.float32(0.08)
    got = oracle.dequant_affine(q, s, b, 8, 128, 64, False)
    g = np.repeat(np.arange(2), 64)
    exact = q.astype(np.float64) * s[:, g].astype(np.float64) + b[:, g].astype(np.float64)
    assert np.array_equal(got, exact.astype(np.float32))


def test_qkv_split_concat_is_input_bitwise():
    seq, qs, ks, vs = 7, 5, 3, 9
    x = synth.normal(5, (seq, qs + ks + vs))
    bits = x.view(np.uint32).copy()
    bits[0, 0] = 0x7FC00123  # a NaN with a payload
    bits[3, 6] = 0xFFC0BEEF
    x = bits.view(np.float32)
    q, k, v = oracle.qkv_split(x, seq, qs, ks, vs)
    back = np.concatenate([q, k, v], axis=1)
    assert np.array_equal(back.view(np.uint32), bits)
    assert np.array_equal(q.view(np.uint32), bits[:, :qs])
    assert np.array_equal(v.view(np.uint32), bits[:, qs + ks:])


def _af4_golden_inputs(N, K):
    r = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    codes = ((3 * k + k // 16 + r) % 16).astype(np.uint8)
    h = np.arange(K // 64)[None, :]
    sb = (0x3C00 + 16 * r + h).astype(np.uint16)
    bb = (0xBC00 + 16 * r + h).astype(np.uint16)
    return codes, sb, bb


def test_af4_g64_golden_words():
    fx = _load("af4_g64.json")
    N, K = fx["N"], fx["K"]
    codes, sb, bb = _af4_golden_inputs(N, K)
    plane, meta = oracle.prepare_af4_g64(codes, sb, bb, N, K)
    assert plane.size == N * K // 8 and meta.size == N * K // 64
    for item in fx["plane"]:
        assert plane[item["index"]] == int(item["word"], 16), item
    for item in fx["metadata"]:
        assert meta[item["index"]] == int(item["word"], 16), item


@pytest.mark.parametrize("N,K", [(192, 256), (64, 64), (320, 1088), (128, 4096)])
def test_af4_g64_layout_is_a_permutation(N, K):
    """Every code lands in exactly one nibble: unpacking returns the input, and
    the plane holds each row's code multiset."""
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 16, (N, K), dtype=np.uint8)
    sb = rng.integers(0, 1 << 16, (N, K // 64), dtype=np.uint16)
    bb = rng.integers(0, 1 << 16, (N, K // 64), dtype=np.uint16)
    plane, meta = oracle.prepare_af4_g64(codes, sb, bb, N, K)
    c2, s2, b2 = oracle.af4_unpack(plane, meta, N, K)
    assert np.array_equal(c2, codes) and np.array_equal(s2, sb) and np.array_equal(b2, bb)
    # The last row's words (the last 64-row block) hold only that row's codes.
    r = N - 1
    words = plane.reshape(N // 64, K // 32, 64, 4)[r // 64, :, r % 64, :].ravel()
    nib = np.concatenate([(words >> (4 * i)) & 15 for i in range(8)])
    assert np.array_equal(np.bincount(nib, minlength=16), np.bincount(codes[r], minlength=16))


def test_af4_bf16_decoder_golden():
    fx = _load("af4_g64.json")
    bits = np.array([int(i["bits"], 16) for i in fx["bf16"]], dtype=np.uint16)
    got = oracle.bf16_to_float_array(bits)
    for g, item in zip(got, fx["bf16"]):
        assert float(g) == item["value"], item


def test_af4_bf16_decoder_matches_torch():
    torch = pytest.importorskip("torch")
    bits = np.arange(0, 1 << 16, 97, dtype=np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # finite values only
    got = oracle.bf16_to_float_array(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
