"""Quantized GEMV with fused dequantization for GB300 (sm_103a).

The compute lives in the CUDA library libqgemv.so (C ABI in include/qgemv.h);
this module is a thin ctypes binding over it with the same names. It only
marshals arguments: torch supplies device memory and the current stream,
every step of the computation runs in the library's kernels. The library is
loaded on first use, and every call raises if it has not been built or no
CUDA device is present: there is no CPU fallback.

Workspace: calls that need device scratch (split-K partial sums) get it from
a torch buffer per (device, stream) that grows on demand, unless the caller
passes one. Calls on different streams therefore never share scratch; calls
on one stream are ordered by the stream.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemv.so")

QG_OK, QG_ERR_INVALID_ARG, QG_ERR_UNSUPPORTED, QG_ERR_MISALIGNED = 0, 1, 2, 3
QG_ERR_CUDA, QG_ERR_WORKSPACE, QG_ERR_DEVICE = 4, 5, 6
QG_OP_Q4_0, QG_OP_DUAL_Q4_0, QG_OP_Q4_K, QG_OP_AFFINE, QG_OP_AF4_G64 = 0, 1, 2, 3, 4
QG_OP_DUAL_Q4_0_HOST = 5
QG_OPT_PDL = 1
QG_OPT_PREFILL_MIN_M = 2
QG_OPT_STREAM, QG_OPT_STREAM_WARPS, QG_OPT_STREAM_SLOTS = 3, 4, 5
QG_OPT_STAGES_AHEAD = 6
QG_OPT_STAGED_WARPS = 7
QG_OPT_PREFILL_FOLD = 8
QG_OPT_XREG = 9
QG_OPT_XREG_AHEAD = 10
QG_OPT_XREG_WARPS = 11
QG_OPT_XREG_CTAS = 12

EXPORTS = ("qgemv_q4_0", "qgemv_dual_q4_0", "qgemv_q4_k", "qmm_affine", "qkv_split",
           "dequant_q4_0", "dequant_q4_k", "dequant_affine", "qg_workspace_size",
           "qg_status_string", "qg_last_cuda_error", "qg_device_error",
           "qg_selftest_wait_timeout", "qg_set_option", "qg_get_option",
           "qgemv_q4_k_noalloc", "qg_prepare_af4_g64", "qmm_af4_g64", "qgemv_dual_q4_0_host")

_LIB = None
_LOCK = threading.Lock()


class QGError(RuntimeError):
    def __init__(self, what: str, status: int):
        self.status = status
        msg = f"{what}: {status_string(status)}"
        if status == QG_ERR_CUDA:
            msg += f" (cudaError {lib().qg_last_cuda_error()})"
        super().__init__(msg)


def lib():
    """The loaded library (ctypes.CDLL), typed. Raises if it was not built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        P, I64, I, SZ = C.c_void_p, C.c_int64, C.c_int, C.c_size_t
        sig = {
            "qgemv_q4_0": [P, P, P, I64, I64, I64, P, SZ, P],
            "qgemv_dual_q4_0": [P, P, P, P, P, I64, I64, I64, P, SZ, P],
            "qgemv_dual_q4_0_host": [P, P, P, P, P, I64, I64, I64, P, SZ, P],
            "qgemv_q4_k": [P, P, P, I64, I64, I64, P, SZ, P],
            "qmm_affine": [P, P, P, P, P, I64, I64, I64, I, I, P, SZ, P],
            "qkv_split": [P, P, P, P, I64, I64, I64, I64, P],
            "dequant_q4_0": [P, P, I64, I64, P],
            "dequant_q4_k": [P, P, I64, I64, P],
            "dequant_affine": [P, P, P, P, I64, I64, I, I, P],
            "qg_workspace_size": [I, I64, I64, I64, I, I, C.POINTER(SZ)],
            "qg_status_string": [I],
            "qg_last_cuda_error": [],
            "qg_device_error": [I, C.POINTER(C.c_uint)],
            "qg_selftest_wait_timeout": [I64, P],
            "qg_set_option": [I, I64],
            "qg_get_option": [I, C.POINTER(I64)],
            "qgemv_q4_k_noalloc": [P, P, P, I64, I64, I64, P],
            "qg_prepare_af4_g64": [P, P, P, P, P, I64, I64, P],
            "qmm_af4_g64": [P, P, P, P, I64, I64, I64, P, SZ, P],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = C.c_char_p if name == "qg_status_string" else C.c_int
        _LIB = L
        return L


def status_string(status: int) -> str:
    return lib().qg_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != QG_OK:
        raise QGError(what, rc)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _host(t: torch.Tensor, name: str, dtype) -> int:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# --------------------------------------------------------------- workspace
_WS = {}


def workspace_size(op: int, M: int, N: int, K: int, group_size: int = 0, packed: int = 0) -> int:
    n = C.c_size_t(0)
    _check(lib().qg_workspace_size(op, M, N, K, group_size, packed, C.byref(n)), "qg_workspace_size")
    return int(n.value)


def _workspace(op, M, N, K, gs, packed, device, workspace, stream):
    need = workspace_size(op, M, N, K, gs, packed)
    if workspace is not None:
        return _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    if need == 0:
        return None, 0
    # One buffer per (device, stream): two calls on different streams may run
    # at the same time and must not share split-K scratch.
    key = (torch.device(device).index, stream)
    with _LOCK:
        buf = _WS.get(key)
        if buf is None or buf.numel() < need:
            buf = torch.empty(need, dtype=torch.uint8, device=device)
            _WS[key] = buf
    return buf.data_ptr(), buf.numel()


# ------------------------------------------------------------------- calls
def qgemv_q4_0(w, x, y=None, *, N=None, workspace=None, stream=None):
    """y[M,N] = x[M,K] . dequant_q4_0(w)^T. w: uint8 Q4_0 bytes of N rows."""
    M, K = x.shape
    N = N if N is not None else w.numel() // (K // 32 * 18)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = _stream(stream)
    ws, wsb = _workspace(QG_OP_Q4_0, M, N, K, 0, 0, x.device, workspace, st)
    _check(lib().qgemv_q4_0(_dev(w, "w", torch.uint8), _dev(x, "x", torch.float32),
                            _dev(y, "y", torch.float32), M, N, K, ws, wsb, st),
           "qgemv_q4_0")
    return y


def qgemv_dual_q4_0(w_a, w_b, x, y_a=None, y_b=None, *, N=None, workspace=None, stream=None):
    """(y_a, y_b) = (x . dequant(w_a)^T, x . dequant(w_b)^T) in one launch."""
    M, K = x.shape
    N = N if N is not None else w_a.numel() // (K // 32 * 18)
    if y_a is None:
        y_a = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if y_b is None:
        y_b = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = _stream(stream)
    ws, wsb = _workspace(QG_OP_DUAL_Q4_0, M, N, K, 0, 0, x.device, workspace, st)
    _check(lib().qgemv_dual_q4_0(_dev(w_a, "w_a", torch.uint8), _dev(w_b, "w_b", torch.uint8),
                                 _dev(x, "x", torch.float32), _dev(y_a, "y_a", torch.float32),
                                 _dev(y_b, "y_b", torch.float32), M, N, K, ws, wsb,
                                 st), "qgemv_dual_q4_0")
    return y_a, y_b


def qgemv_dual_q4_0_host(w_a, w_b, x, y_a=None, y_b=None, *, N=None, workspace=None,
                         stream=None):
    """qgemv_dual_q4_0 with x, y_a, y_b in host memory (CPU tensors); returns
    once y_a and y_b hold the result. Page-locked buffers (pin_memory()) are
    read and written in place for M <= 2; other buffers pass through device
    staging. New outputs are page-locked when x is."""
    M, K = x.shape
    N = N if N is not None else w_a.numel() // (K // 32 * 18)
    pin = x.is_pinned()
    if y_a is None:
        y_a = torch.empty((M, N), dtype=torch.float32, pin_memory=pin)
    if y_b is None:
        y_b = torch.empty((M, N), dtype=torch.float32, pin_memory=pin)
    st = _stream(stream)
    ws, wsb = _workspace(QG_OP_DUAL_Q4_0_HOST, M, N, K, 0, 0, w_a.device, workspace, st)
    _check(lib().qgemv_dual_q4_0_host(_dev(w_a, "w_a", torch.uint8), _dev(w_b, "w_b", torch.uint8),
                                      _host(x, "x", torch.float32), _host(y_a, "y_a", torch.float32),
                                      _host(y_b, "y_b", torch.float32), M, N, K, ws, wsb, st),
           "qgemv_dual_q4_0_host")
    return y_a, y_b


def qgemv_q4_k(w, x, y=None, *, N=None, workspace=None, stream=None):
    """y[M,N] = x[M,K] . dequant_q4_k(w)^T. w: uint8 Q4_K bytes of N rows."""
    M, K = x.shape
    N = N if N is not None else w.numel() // (K // 256 * 144)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = _stream(stream)
    ws, wsb = _workspace(QG_OP_Q4_K, M, N, K, 0, 0, x.device, workspace, st)
    _check(lib().qgemv_q4_k(_dev(w, "w", torch.uint8), _dev(x, "x", torch.float32),
                            _dev(y, "y", torch.float32), M, N, K, ws, wsb, st),
           "qgemv_q4_k")
    return y


def qgemv_q4_k_noalloc(w, x, y=None, *, N=None, stream=None):
    """qgemv_q4_k without a caller workspace: split-K scratch lives in a fixed
    4 MiB device array inside the library (see include/qgemv.h)."""
    M, K = x.shape
    N = N if N is not None else w.numel() // (K // 256 * 144)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check(lib().qgemv_q4_k_noalloc(_dev(w, "w", torch.uint8), _dev(x, "x", torch.float32),
                                    _dev(y, "y", torch.float32), M, N, K, _stream(stream)),
           "qgemv_q4_k_noalloc")
    return y


def qmm_affine(x, q, scales, biases, group_size, packed, y=None, *, workspace=None, stream=None):
    """y = x . dequant_affine(q, scales, biases)^T; q uint8 codes ([N,K] or [N,K/2])."""
    M, K = x.shape
    N = scales.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = _stream(stream)
    ws, wsb = _workspace(QG_OP_AFFINE, M, N, K, group_size, int(packed), x.device, workspace, st)
    _check(lib().qmm_affine(_dev(x, "x", torch.float32), _dev(q, "q", torch.uint8),
                            _dev(scales, "scales", torch.float32),
                            _dev(biases, "biases", torch.float32), _dev(y, "y", torch.float32),
                            M, N, K, int(group_size), int(packed), ws, wsb, st),
           "qmm_affine")
    return y


def prepare_af4_g64(codes, scales, biases, *, stream=None):
    """(plane, metadata) of the prepared AF4-g64 layout (int32 tensors holding
    the u32 words): codes uint8 [N, K] (0..15), scales and biases bfloat16
    [N, K/64]."""
    N, K = codes.shape
    plane = torch.empty(N * K // 8, dtype=torch.int32, device=codes.device)
    meta = torch.empty(N * K // 64, dtype=torch.int32, device=codes.device)
    _check(lib().qg_prepare_af4_g64(_dev(codes, "codes", torch.uint8),
                                    _dev(scales, "scales", torch.bfloat16),
                                    _dev(biases, "biases", torch.bfloat16), plane.data_ptr(),
                                    meta.data_ptr(), N, K, _stream(stream)), "qg_prepare_af4_g64")
    return plane, meta


def qmm_af4_g64(x, plane, metadata, N, y=None, *, workspace=None, stream=None):
    """y[M,N] = x[M,K] . w^T from the prepared AF4-g64 layout (M <= 32; no workspace)."""
    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = _stream(stream)
    ws, wsb = _workspace(QG_OP_AF4_G64, M, N, K, 0, 0, x.device, workspace, st)
    _check(lib().qmm_af4_g64(_dev(x, "x", torch.float32), _dev(plane, "plane", torch.int32),
                             _dev(metadata, "metadata", torch.int32), _dev(y, "y", torch.float32),
                             M, N, K, ws, wsb, st), "qmm_af4_g64")
    return y


def qkv_split(qkv, q_sp, k_sp, v_sp, q=None, k=None, v=None, *, stream=None):
    """Split [seq, q_sp+k_sp+v_sp] f32 into q [seq,q_sp], k [seq,k_sp], v [seq,v_sp]."""
    seq = qkv.shape[0]
    dev = qkv.device
    q = torch.empty((seq, q_sp), dtype=torch.float32, device=dev) if q is None else q
    k = torch.empty((seq, k_sp), dtype=torch.float32, device=dev) if k is None else k
    v = torch.empty((seq, v_sp), dtype=torch.float32, device=dev) if v is None else v
    _check(lib().qkv_split(_dev(qkv, "qkv", torch.float32), _dev(q, "q", torch.float32),
                           _dev(k, "k", torch.float32), _dev(v, "v", torch.float32), seq, q_sp,
                           k_sp, v_sp, _stream(stream)), "qkv_split")
    return q, k, v


def dequant_q4_0(w, N, K, out=None, *, stream=None):
    out = torch.empty((N, K), dtype=torch.float32, device=w.device) if out is None else out
    _check(lib().dequant_q4_0(_dev(w, "w", torch.uint8), _dev(out, "out", torch.float32), N, K,
                              _stream(stream)), "dequant_q4_0")
    return out


def dequant_q4_k(w, N, K, out=None, *, stream=None):
    out = torch.empty((N, K), dtype=torch.float32, device=w.device) if out is None else out
    _check(lib().dequant_q4_k(_dev(w, "w", torch.uint8), _dev(out, "out", torch.float32), N, K,
                              _stream(stream)), "dequant_q4_k")
    return out


def dequant_affine(q, scales, biases, N, K, group_size, packed, out=None, *, stream=None):
    out = torch.empty((N, K), dtype=torch.float32, device=q.device) if out is None else out
    _check(lib().dequant_affine(_dev(q, "q", torch.uint8), _dev(scales, "scales", torch.float32),
                                _dev(biases, "biases", torch.float32),
                                _dev(out, "out", torch.float32), N, K, int(group_size),
                                int(packed), _stream(stream)), "dequant_affine")
    return out


def device_error(clear: bool = True) -> int:
    """Synchronize and return (optionally clearing) the device error word."""
    code = C.c_uint(0)
    rc = lib().qg_device_error(int(clear), C.byref(code))
    if rc not in (QG_OK, QG_ERR_DEVICE):
        raise QGError("qg_device_error", rc)
    return int(code.value)


def selftest_wait_timeout(timeout_ns: int, *, stream=None):
    _check(lib().qg_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
           "qg_selftest_wait_timeout")


def set_option(option: int, value: int):
    """qg_set_option: e.g. set_option(QG_OPT_PDL, 1) (see include/qgemv.h)."""
    _check(lib().qg_set_option(int(option), int(value)), "qg_set_option")


def get_option(option: int) -> int:
    v = C.c_int64(0)
    _check(lib().qg_get_option(int(option), C.byref(v)), "qg_get_option")
    return int(v.value)
