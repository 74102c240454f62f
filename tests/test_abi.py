"""The C-ABI library builds, loads and exports every symbol include/qgemv.h
declares; host-side validation rejects bad arguments without touching a GPU
(CPU only: no compute call is made)."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_gemv_dequant_gb300 import _build
    path = _build.build()
    return C.CDLL(path)


def declared_symbols():
    with open(os.path.join(ROOT, "include", "qgemv.h")) as f:
        text = f.read()
    return re.findall(r"QG_API\s+(?:const\s+)?\w+\*?\s+(\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    for n in ("qgemv_q4_0", "qgemv_dual_q4_0", "qgemv_q4_k", "qmm_affine", "qkv_split",
              "dequant_q4_0", "dequant_q4_k", "dequant_affine"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_binding_names_match_header():
    import bit_quantized_gemv_dequant_gb300 as qg
    assert set(qg.EXPORTS) == set(declared_symbols())


def test_status_strings(lib):
    lib.qg_status_string.restype = C.c_char_p
    assert lib.qg_status_string(0) == b"ok"
    assert lib.qg_status_string(1) == b"invalid argument"
    assert lib.qg_status_string(99) == b"unknown status"


def test_validation_needs_no_gpu(lib):
    P, I64 = C.c_void_p, C.c_int64
    f = lib.qgemv_q4_0
    f.argtypes = [P, P, P, I64, I64, I64, P, C.c_size_t, P]
    fake = 0x10000
    # zero M, K not a multiple of 32, NULL weight, output aliasing input
    assert f(fake, fake + 4096, fake + 8192, 0, 4, 64, None, 0, None) == 1
    assert f(fake, fake + 4096, fake + 8192, 1, 4, 48, None, 0, None) == 1
    assert f(None, fake + 4096, fake + 8192, 1, 4, 64, None, 0, None) == 1
    assert f(fake, fake + 4096, fake + 4096, 1, 4, 64, None, 0, None) == 1
    assert f(fake, fake + 4098, fake + 8192, 1, 4, 64, None, 0, None) == 3  # x misaligned
    g = lib.qmm_affine
    g.argtypes = [P, P, P, P, P, I64, I64, I64, C.c_int, C.c_int, P, C.c_size_t, P]
    assert g(fake, fake + 4096, fake + 8192, fake + 12288, fake + 16384, 1, 4, 64, 48, 0,
             None, 0, None) == 1  # group size not a power of two
    assert g(fake, fake + 4096, fake + 8192, fake + 12288, fake + 16384, 1, 4, 64, 2048, 0,
             None, 0, None) == 1  # group size above 1024
    assert g(fake, fake + 4096, fake + 8192, fake + 12288, fake + 16384, 1, 4, 63, 64, 1,
             None, 0, None) == 1
    h = lib.qkv_split
    h.argtypes = [P, P, P, P, I64, I64, I64, I64, P]
    assert h(fake, fake + 4096, fake + 8192, fake + 12288, 4, 0, 1, 1, None) == 1
    assert h(fake, fake + 4096, fake + 8192, fake + 12288, 4, 2**62, 2**62, 1, None) == 1
    k = lib.qgemv_q4_k
    k.argtypes = [P, P, P, I64, I64, I64, P, C.c_size_t, P]
    assert k(fake, fake + 4096, fake + 8192, 1, 4, 128, None, 0, None) == 1  # K % 256
    a = lib.qmm_af4_g64
    a.argtypes = [P, P, P, P, I64, I64, I64, P, C.c_size_t, P]
    x, pl, me, y = fake, fake + 65536, fake + 131072, fake + 196608
    assert a(x, pl, me, y, 33, 64, 64, None, 0, None) == 1      # M > 32
    assert a(x, pl, me, y, 1, 96, 64, None, 0, None) == 1       # N % 64
    assert a(x, pl, me, y, 1, 64, 96, None, 0, None) == 1       # K % 64
    assert a(None, pl, me, y, 1, 64, 64, None, 0, None) == 1
    assert a(x, pl + 4, me, y, 1, 64, 64, None, 0, None) == 3   # plane not 16-byte aligned
    assert a(x, pl, me, x, 1, 64, 64, None, 0, None) == 1       # y overlaps x
    pr = lib.qg_prepare_af4_g64
    pr.argtypes = [P, P, P, P, P, I64, I64, P]
    assert pr(fake, fake + 8192, fake + 12288, pl, me, 64, 96, None) == 1   # K % 64
    assert pr(fake, fake + 8192, fake + 12288, pl + 8, me, 64, 64, None) == 3
    assert pr(fake, None, fake + 12288, pl, me, 64, 64, None) == 1
    ws = C.c_size_t(7)
    lib.qg_workspace_size.argtypes = [C.c_int, I64, I64, I64, C.c_int, C.c_int,
                                      C.POINTER(C.c_size_t)]
    assert lib.qg_workspace_size(4, 32, 64, 128, 0, 0, C.byref(ws)) == 0 and ws.value == 0
    assert lib.qg_workspace_size(4, 33, 64, 128, 0, 0, C.byref(ws)) == 1


def test_launch_options_round_trip_and_validation(lib):
    """qg_set_option / qg_get_option need no GPU: values round-trip, and values
    outside each option's documented range are refused."""
    lib.qg_set_option.argtypes = [C.c_int, C.c_int64]
    lib.qg_get_option.argtypes = [C.c_int, C.POINTER(C.c_int64)]
    get = lambda o: (lambda v: (lib.qg_get_option(o, C.byref(v)), v.value))(C.c_int64())
    cases = {1: ([0, 1, 2], [3, -1]),         # QG_OPT_PDL
             2: ([1, 64], [0]),               # QG_OPT_PREFILL_MIN_M
             3: ([0, 1, 2], [3, -1]),         # QG_OPT_STREAM
             4: ([0, 1, 8], [9, -1]),         # QG_OPT_STREAM_WARPS
             5: ([0, 2, 8], [1, 9]),          # QG_OPT_STREAM_SLOTS
             6: ([0, 1, 64], [65, -1]),       # QG_OPT_STAGES_AHEAD
             7: ([0, 8], [4, 16]),            # QG_OPT_STAGED_WARPS
             8: ([0, 1], [2, -1]),            # QG_OPT_PREFILL_FOLD
             9: ([0, 1], [2, -1]),            # QG_OPT_XREG
             10: ([0, 1, 16], [17, -1]),      # QG_OPT_XREG_AHEAD
             11: ([4, 8, 16, 0], [2, 12, -1]),  # QG_OPT_XREG_WARPS
             12: ([2, 4, 1, 0], [-1, 5])}     # QG_OPT_XREG_CTAS
    for opt, (good, bad) in cases.items():
        rc, old = get(opt)
        assert rc == 0
        try:
            for v in good:
                assert lib.qg_set_option(opt, v) == 0
                assert get(opt) == (0, v)
            for v in bad:
                assert lib.qg_set_option(opt, v) == 1  # QG_ERR_INVALID_ARG
                assert get(opt)[1] == good[-1]
        finally:
            assert lib.qg_set_option(opt, old) == 0
    assert lib.qg_set_option(99, 0) == 1
