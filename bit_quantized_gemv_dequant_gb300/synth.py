"""Seeded synthetic inputs (the input recipe shared by tests and the benchmark).

This module only draws random numbers and encodes the drawn weights into the
byte formats the library consumes. It computes no dequantization and no
product: that arithmetic belongs to the CUDA kernels on one side and to the
independent CPU oracle on the other, and neither uses anything from here but
the arrays it returns.

Random numbers come from numpy's PCG64 generator, one stream per
(seed, tensor) pair. Weight encoders follow the workload recipe:

* Q4_0 (fused_dual_proj_q4_0.rs, mlx-native 0.9.1: 18-byte blocks of fp16 d
  plus 16 nibble bytes along K): per 32-wide block, d = (the element of
  largest magnitude, lowest index on ties) / -8 in f32, stored as fp16
  (round to nearest even); q = clamp(round(w / d) + 8, 0, 15) with the f32 d
  and rounding half away from zero; an all-zero block stores d = 0, q = 8.
  Byte 2+j holds element j (low nibble) and element 16+j (high nibble).
* Q4_K (q4_k_gemv_v2.rs, ferrum-kernels 0.7.7: 144-byte super-blocks of
  256 weights): per 32-wide sub-block lo = min(0, min w), hi = max w,
  scale = (hi - lo) / 15, min = -lo; d = max scale / 63 and dmin = max min / 63
  stored as fp16; sc = clamp(round(scale / d), 0, 63), m = clamp(round(min /
  dmin), 0, 63) and q = clamp(round((w + dmin*m) / (d*sc)), 0, 15) with the
  stored d, dmin (a zero divisor gives 0). Field layout: d, dmin, 12 bytes of
  6-bit pairs (GGUF packing), 128 nibble bytes in four 32-byte chunks whose
  low nibbles are sub-block 2c and high nibbles sub-block 2c+1.
* Affine (qmm_affine.rs, mlx-native 0.21.1): codes, scales and biases are
  drawn directly; pack_nibbles is the byte view of pack_b4_to_u32 (element 2i
  in the low nibble of byte i).
"""
from __future__ import annotations

import numpy as np

# Tensor ids used to derive per-tensor seeds: seed = 1000 * case + tensor id.
T_W, T_W_B, T_X, T_Q, T_S, T_B, T_QKV = 1, 2, 3, 4, 5, 6, 7


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def normal(seed: int, shape, sigma: float = 1.0) -> np.ndarray:
    a = rng(seed).standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    return a


def uniform(seed: int, shape, lo: float, hi: float) -> np.ndarray:
    a = rng(seed).random(size=shape, dtype=np.float32)
    return (np.float32(lo) + a * np.float32(hi - lo)).astype(np.float32)


def codes(seed: int, shape, bits: int = 4) -> np.ndarray:
    return rng(seed).integers(0, 1 << bits, size=shape, dtype=np.uint8)


def round_half_away(v: np.ndarray) -> np.ndarray:
    """Round f32 values to the nearest integer, halves away from zero (exact)."""
    v = np.asarray(v, dtype=np.float32)
    t = np.trunc(v)
    frac = v - t  # exact for |v| < 2^23
    return t + np.where(np.abs(frac) >= np.float32(0.5), np.sign(v), np.float32(0.0))


# ----------------------------------------------------------------------- Q4_0
def q4_0_from_parts(d_bits: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Assemble Q4_0 bytes from fp16 d bits [N, nb] and codes [N, nb, 32]."""
    N, nb = d_bits.shape
    out = np.empty((N, nb, 18), dtype=np.uint8)
    d_bits = np.asarray(d_bits, dtype=np.uint16)
    q = np.asarray(q, dtype=np.uint8)
    out[..., 0] = (d_bits & 0xFF).astype(np.uint8)
    out[..., 1] = (d_bits >> 8).astype(np.uint8)
    out[..., 2:] = q[..., :16] | (q[..., 16:] << 4)
    return out.reshape(N, nb * 18)


def quantize_q4_0(W: np.ndarray) -> np.ndarray:
    """W f32 [N, K] (K % 32 == 0) -> Q4_0 bytes [N, K/32*18]."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % 32 == 0
    blk = W.reshape(N, K // 32, 32)
    idx = np.argmax(np.abs(blk), axis=2)  # first occurrence on ties
    amax = np.take_along_axis(blk, idx[..., None], axis=2)[..., 0]
    d = (amax / np.float32(-8.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = round_half_away(blk / d[..., None])
    q = np.where(d[..., None] == 0, np.float32(8.0), np.clip(r + 8.0, 0.0, 15.0))
    return q4_0_from_parts(d.astype(np.float16).view(np.uint16), q.astype(np.uint8))


# ----------------------------------------------------------------------- Q4_K
def pack_q4_k_scales(sc: np.ndarray, m: np.ndarray) -> np.ndarray:
    """6-bit sc, m [..., 8] -> 12 packed bytes [..., 12] (GGUF packing)."""
    sc = np.asarray(sc, dtype=np.uint8)
    m = np.asarray(m, dtype=np.uint8)
    s = np.zeros(sc.shape[:-1] + (12,), dtype=np.uint8)
    for i in range(4):
        s[..., i] = (sc[..., i] & 63) | ((sc[..., i + 4] >> 4) << 6)
        s[..., i + 4] = (m[..., i] & 63) | ((m[..., i + 4] >> 4) << 6)
        s[..., i + 8] = (sc[..., i + 4] & 15) | ((m[..., i + 4] & 15) << 4)
    return s


def q4_k_from_parts(d_bits, dmin_bits, sc, m, q) -> np.ndarray:
    """Assemble Q4_K bytes from fp16 bits [N, nb], sc/m [N, nb, 8], q [N, nb, 256]."""
    d_bits = np.asarray(d_bits, dtype=np.uint16)
    dmin_bits = np.asarray(dmin_bits, dtype=np.uint16)
    N, nb = d_bits.shape
    out = np.empty((N, nb, 144), dtype=np.uint8)
    out[..., 0] = (d_bits & 0xFF).astype(np.uint8)
    out[..., 1] = (d_bits >> 8).astype(np.uint8)
    out[..., 2] = (dmin_bits & 0xFF).astype(np.uint8)
    out[..., 3] = (dmin_bits >> 8).astype(np.uint8)
    out[..., 4:16] = pack_q4_k_scales(sc, m)
    q = np.asarray(q, dtype=np.uint8).reshape(N, nb, 4, 64)
    out[..., 16:] = (q[..., :32] | (q[..., 32:] << 4)).reshape(N, nb, 128)
    return out.reshape(N, nb * 144)


def quantize_q4_k(W: np.ndarray) -> np.ndarray:
    """W f32 [N, K] (K % 256 == 0) -> Q4_K bytes [N, K/256*144]."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % 256 == 0
    nb = K // 256
    sub = W.reshape(N, nb, 8, 32)
    lo = np.minimum(np.float32(0.0), sub.min(axis=3))
    hi = sub.max(axis=3)
    scale = ((hi - lo) / np.float32(15.0)).astype(np.float32)
    mins = (-lo).astype(np.float32)
    d16 = (scale.max(axis=2) / np.float32(63.0)).astype(np.float16)
    dmin16 = (mins.max(axis=2) / np.float32(63.0)).astype(np.float16)
    d = d16.astype(np.float32)
    dmin = dmin16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d[..., None] > 0, round_half_away(scale / d[..., None]), 0.0)
        m = np.where(dmin[..., None] > 0, round_half_away(mins / dmin[..., None]), 0.0)
    sc = np.clip(sc, 0, 63).astype(np.uint8)
    m = np.clip(m, 0, 63).astype(np.uint8)
    ds = (d[..., None] * sc.astype(np.float32)).astype(np.float32)
    dm = (dmin[..., None] * m.astype(np.float32)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = round_half_away((sub + dm[..., None]) / ds[..., None])
    qf = np.where(ds[..., None] > 0, qf, 0.0)
    q = np.clip(qf, 0, 15).astype(np.uint8).reshape(N, nb, 256)
    return q4_k_from_parts(d16.view(np.uint16), dmin16.view(np.uint16), sc, m, q)


# --------------------------------------------------------------------- affine
def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Codes u8 [N, K] (K even, values < 16) -> packed bytes [N, K/2]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    return (q[:, 0::2] & 0x0F) | ((q[:, 1::2] & 0x0F) << 4)


# ------------------------------------------------------------------ workloads
def q4_0_case(case: int, N: int, K: int, M: int, dual: bool = False) -> dict:
    """W ~ N(0, 0.02^2) encoded as Q4_0; x ~ N(0, 1) of shape [M, K]."""
    out = {"w": quantize_q4_0(normal(1000 * case + T_W, (N, K), 0.02)),
           "x": normal(1000 * case + T_X, (M, K))}
    if dual:
        out["w_b"] = quantize_q4_0(normal(1000 * case + T_W_B, (N, K), 0.02))
    return out


def q4_k_case(case: int, N: int, K: int, M: int) -> dict:
    """W ~ N(0, 0.02^2) encoded as Q4_K; x ~ N(0, 1) of shape [M, K]."""
    return {"w": quantize_q4_k(normal(1000 * case + T_W, (N, K), 0.02)),
            "x": normal(1000 * case + T_X, (M, K))}


def affine_case(case: int, N: int, K: int, M: int, gs: int) -> dict:
    """q ~ U{0..15}, s ~ U(0.001, 0.01), b ~ U(-0.08, 0), x ~ N(0, 1)."""
    q = codes(1000 * case + T_Q, (N, K))
    return {"q": q, "q_packed": pack_nibbles(q),
            "s": uniform(1000 * case + T_S, (N, K // gs), 0.001, 0.01),
            "b": uniform(1000 * case + T_B, (N, K // gs), -0.08, 0.0),
            "x": normal(1000 * case + T_X, (M, K))}


def bf16_bits(v: np.ndarray) -> np.ndarray:
    """f32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def af4_case(case: int, N: int, K: int, M: int) -> dict:
    """AF4-g64 inputs: codes U{0..15}, bf16 scales ~ U(0.001, 0.01) and
    biases ~ U(-0.08, 0) per 64-group (as bit patterns), x ~ N(0, 1)."""
    return {"q": codes(1000 * case + T_Q, (N, K)),
            "s_bits": bf16_bits(uniform(1000 * case + T_S, (N, K // 64), 0.001, 0.01)),
            "b_bits": bf16_bits(uniform(1000 * case + T_B, (N, K // 64), -0.08, 0.0)),
            "x": normal(1000 * case + T_X, (M, K))}


def qkv_case(case: int, seq: int, q_sp: int, k_sp: int, v_sp: int) -> np.ndarray:
    return normal(1000 * case + T_QKV, (seq, q_sp + k_sp + v_sp))
