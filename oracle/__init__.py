"""Plain CPU oracle (test infrastructure only).

This package wraps oracle/oracle.c through ctypes. It is the independent
reference the CUDA library is checked against: it shares no code with the
product, and the product never imports it. Only tests/, the smoke check in
__graft_entry__.py and the CPU-baseline leg of bench.py may use it.

Every function dequantizes exactly as the format defines and accumulates in
f64; the GEMV functions also return bound = sum_k |x_k * w_k| per output, the
scale of the parity tolerance. See oracle.c for the definitions and the
readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import build as _build

_LIB = None

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_i64 = C.c_int64


def _bind(path: str):
    L = C.CDLL(path)
    L.orc_half_to_float.argtypes = [C.c_uint16]
    L.orc_half_to_float.restype = C.c_float
    L.orc_q4_0_block.argtypes = [_u8p, _f32p]
    L.orc_q4_0_block.restype = None
    L.orc_dequant_q4_0.argtypes = [_u8p, _i64, _i64, _f32p]
    L.orc_dequant_q4_0.restype = None
    L.orc_q4_k_scale_min.argtypes = [_u8p, C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_int)]
    L.orc_q4_k_scale_min.restype = None
    L.orc_q4_k_block.argtypes = [_u8p, _f32p]
    L.orc_q4_k_block.restype = None
    L.orc_dequant_q4_k.argtypes = [_u8p, _i64, _i64, _f32p]
    L.orc_dequant_q4_k.restype = None
    L.orc_dequant_affine.argtypes = [_u8p, _f32p, _f32p, _i64, _i64, C.c_int, C.c_int, _f32p]
    L.orc_dequant_affine.restype = None
    L.orc_gemv_dense.argtypes = [_f32p, _f32p, _i64, _i64, _i64, _f64p, _f64p]
    L.orc_gemv_dense.restype = None
    rows_t = C.c_void_p
    L.orc_gemv_q4_0.argtypes = [_u8p, _f32p, _i64, _i64, _i64, rows_t, _i64, _f64p, _f64p]
    L.orc_gemv_q4_0.restype = C.c_int
    L.orc_gemv_q4_k.argtypes = [_u8p, _f32p, _i64, _i64, _i64, rows_t, _i64, _f64p, _f64p]
    L.orc_gemv_q4_k.restype = C.c_int
    L.orc_qmm_affine.argtypes = [_f32p, _u8p, _f32p, _f32p, _i64, _i64, _i64, C.c_int,
                                 C.c_int, rows_t, _i64, _f64p, _f64p]
    L.orc_qmm_affine.restype = C.c_int
    L.orc_gemv_dual_q4_0.argtypes = [_u8p, _u8p, _f32p, _i64, _i64, _i64, rows_t, _i64,
                                     _f64p, _f64p, _f64p, _f64p]
    L.orc_gemv_dual_q4_0.restype = C.c_int
    L.orc_qkv_split.argtypes = [_u32p, _u32p, _u32p, _u32p, _i64, _i64, _i64, _i64]
    L.orc_qkv_split.restype = None
    _u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
    L.orc_prepare_af4_g64.argtypes = [_u8p, _u16p, _u16p, _i64, _i64, _u32p, _u32p]
    L.orc_prepare_af4_g64.restype = None
    L.orc_af4_unpack.argtypes = [_u32p, _u32p, _i64, _i64, _u8p, _u16p, _u16p]
    L.orc_af4_unpack.restype = None
    L.orc_bf16_to_float.argtypes = [C.c_uint16]
    L.orc_bf16_to_float.restype = C.c_float
    return L


def lib():
    global _LIB
    if _LIB is None:
        _LIB = _bind(_build.build())
    return _LIB


def use_library(path):
    """Point the wrappers at another build of oracle.c (None restores the
    normal one). Used only by the planted-mistake tests."""
    global _LIB
    _LIB = None if path is None else _bind(path)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _rows(rows):
    if rows is None:
        return None, 0, None
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r.ctypes.data_as(C.c_void_p), int(r.size), r


# --------------------------------------------------------------------- formats
def half_to_float(bits: int) -> float:
    return float(lib().orc_half_to_float(int(bits) & 0xFFFF))


def half_to_float_array(bits) -> np.ndarray:
    L = lib()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.empty(flat.size, dtype=np.float32)
    f = L.orc_half_to_float
    for i, h in enumerate(flat.tolist()):
        out[i] = f(h)
    return out.reshape(np.shape(bits))


def q4_0_block(blk) -> np.ndarray:
    out = np.empty(32, dtype=np.float32)
    lib().orc_q4_0_block(_c(blk, np.uint8), out)
    return out


def dequant_q4_0(w: np.ndarray, N: int, K: int) -> np.ndarray:
    out = np.empty((N, K), dtype=np.float32)
    lib().orc_dequant_q4_0(_c(w, np.uint8).ravel(), N, K, out)
    return out


def q4_k_scale_min(scales12, j: int):
    sc, m = C.c_int(), C.c_int()
    lib().orc_q4_k_scale_min(_c(scales12, np.uint8), j, C.byref(sc), C.byref(m))
    return sc.value, m.value


def q4_k_block(blk) -> np.ndarray:
    out = np.empty(256, dtype=np.float32)
    lib().orc_q4_k_block(_c(blk, np.uint8), out)
    return out


def dequant_q4_k(w: np.ndarray, N: int, K: int) -> np.ndarray:
    out = np.empty((N, K), dtype=np.float32)
    lib().orc_dequant_q4_k(_c(w, np.uint8).ravel(), N, K, out)
    return out


def dequant_affine(q, s, b, N: int, K: int, gs: int, packed: bool) -> np.ndarray:
    out = np.empty((N, K), dtype=np.float32)
    lib().orc_dequant_affine(_c(q, np.uint8).ravel(), _c(s, np.float32).ravel(),
                             _c(b, np.float32).ravel(), N, K, gs, int(bool(packed)), out)
    return out


# ----------------------------------------------------------------------- GEMV
def gemv_dense(W, x, M: int, N: int, K: int):
    ref = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    lib().orc_gemv_dense(_c(W, np.float32).ravel(), _c(x, np.float32).ravel(), M, N, K, ref, bound)
    return ref, bound


def _check(rc):
    if rc:
        raise MemoryError("oracle allocation failed")


def gemv_q4_0(w, x, M: int, N: int, K: int, rows=None):
    ref = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    rp, nr, _keep = _rows(rows)
    _check(lib().orc_gemv_q4_0(_c(w, np.uint8).ravel(), _c(x, np.float32).ravel(), M, N, K, rp,
                               nr, ref, bound))
    return ref, bound


def gemv_q4_k(w, x, M: int, N: int, K: int, rows=None):
    ref = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    rp, nr, _keep = _rows(rows)
    _check(lib().orc_gemv_q4_k(_c(w, np.uint8).ravel(), _c(x, np.float32).ravel(), M, N, K, rp,
                               nr, ref, bound))
    return ref, bound


def gemv_dual_q4_0(w_a, w_b, x, M: int, N: int, K: int, rows=None):
    ra = np.zeros((M, N), dtype=np.float64)
    ba = np.zeros((M, N), dtype=np.float64)
    rb = np.zeros((M, N), dtype=np.float64)
    bb = np.zeros((M, N), dtype=np.float64)
    rp, nr, _keep = _rows(rows)
    _check(lib().orc_gemv_dual_q4_0(_c(w_a, np.uint8).ravel(), _c(w_b, np.uint8).ravel(),
                                    _c(x, np.float32).ravel(), M, N, K, rp, nr, ra, ba, rb, bb))
    return (ra, ba), (rb, bb)


def qmm_affine(x, q, s, b, M: int, N: int, K: int, gs: int, packed: bool, rows=None):
    ref = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    rp, nr, _keep = _rows(rows)
    _check(lib().orc_qmm_affine(_c(x, np.float32).ravel(), _c(q, np.uint8).ravel(),
                                _c(s, np.float32).ravel(), _c(b, np.float32).ravel(), M, N, K, gs,
                                int(bool(packed)), rp, nr, ref, bound))
    return ref, bound


# ---------------------------------------------------------------- AF4-g64
def prepare_af4_g64(codes, scales_bits, biases_bits, N: int, K: int):
    """(plane u32 [N*K/8], meta u32 [N*K/64]) of the prepared layout."""
    plane = np.zeros(N * K // 8, dtype=np.uint32)
    meta = np.zeros(N * K // 64, dtype=np.uint32)
    lib().orc_prepare_af4_g64(_c(codes, np.uint8).ravel(), _c(scales_bits, np.uint16).ravel(),
                              _c(biases_bits, np.uint16).ravel(), N, K, plane, meta)
    return plane, meta


def af4_unpack(plane, meta, N: int, K: int):
    """(codes u8 [N, K], scale bits u16 [N, K/64], bias bits u16 [N, K/64])."""
    codes = np.zeros((N, K), dtype=np.uint8)
    sb = np.zeros((N, K // 64), dtype=np.uint16)
    bb = np.zeros((N, K // 64), dtype=np.uint16)
    lib().orc_af4_unpack(_c(plane, np.uint32).ravel(), _c(meta, np.uint32).ravel(), N, K,
                         codes.reshape(-1), sb.reshape(-1), bb.reshape(-1))
    return codes, sb, bb


def bf16_to_float_array(bits) -> np.ndarray:
    f = lib().orc_bf16_to_float
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.empty(flat.size, dtype=np.float32)
    for i, h in enumerate(flat.tolist()):
        out[i] = f(h)
    return out.reshape(np.shape(bits))


def qmm_af4_g64(x, codes, scales_bits, biases_bits, M: int, N: int, K: int, rows=None):
    """The AF4-g64 qmm from its unprepared definition: qmm_affine with group
    size 64 and the bf16 scales and biases taken exactly as f32."""
    s = bf16_to_float_array(scales_bits)
    b = bf16_to_float_array(biases_bits)
    return qmm_affine(x, codes, s, b, M, N, K, 64, False, rows=rows)


def qkv_split(qkv, seq: int, q_sp: int, k_sp: int, v_sp: int):
    src = _c(qkv, np.float32).view(np.uint32).ravel()
    q = np.empty(seq * q_sp, dtype=np.uint32)
    k = np.empty(seq * k_sp, dtype=np.uint32)
    v = np.empty(seq * v_sp, dtype=np.uint32)
    lib().orc_qkv_split(src, q, k, v, seq, q_sp, k_sp, v_sp)
    return (q.view(np.float32).reshape(seq, q_sp), k.view(np.float32).reshape(seq, k_sp),
            v.view(np.float32).reshape(seq, v_sp))


# ------------------------------------------------------------------ tolerance
# Parity bar for the f32 CUDA-core paths: |y - ref| <= REL * bound + ABS, with
# bound = sum_k |x_k w_k| (f64). The tensor-core prefill path uses REL_TC.
REL = 1e-5
ABS = 1e-6
REL_TC = 2e-3


def within(y, ref, bound, rel: float = REL, abs_: float = ABS):
    """Element-wise pass mask and the worst ratio |y-ref| / (rel*bound+abs)."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - ref)
    lim = rel * bound + abs_
    ok = err <= lim
    ratio = float(np.max(err / lim)) if err.size else 0.0
    return ok, ratio
