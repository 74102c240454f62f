"""GPU test of qgemv_q4_k_noalloc, the Q4_K GEMV for callers that cannot
allocate device memory (it takes its split-K scratch from a fixed array in the
library instead of a caller workspace).

Collected last on purpose: a run that stops at the first failure has run
every other test before this one. It also passes on its own in a fresh
process: it builds all its inputs itself and needs no state from other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_parity, to_dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    # Both shapes need split-K scratch (x for M rows of K = 12288 does not fit
    # in shared memory), so the fixed array is really used, twice in a row.
    shapes = [(8, 96, 12288), (4, 200, 12288)]
    for i, (M, N, K) in enumerate(shapes):
        assert qg.workspace_size(qg.QG_OP_Q4_K, M, N, K) > 0
        c = synth.q4_k_case(3000 + i, N, K, M)
        w, x = to_dev(c["w"]), to_dev(c["x"])
        y_new = qg.qgemv_q4_k_noalloc(w, x, N=N)
        y_old = qg.qgemv_q4_k(w, x, N=N)
        torch.cuda.synchronize()
        # Same tolerance as every GEMV parity test, with the existing entry
        # point's output as the reference value and the oracle's sum |x w| as
        # the scale.
        _, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
        assert_parity(y_new, y_old.cpu().numpy().astype(np.float64), bound,
                      what=f"no-alloc vs workspace call {i}")
        ref, _ = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
        assert_parity(y_new, ref, bound, what=f"no-alloc vs oracle call {i}")
    assert qg.device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 3 slices x 8 rows x 65536 outputs x 4 bytes = 6 MiB > 4 MiB: refused with
    # QG_ERR_WORKSPACE before anything is enqueued (the pointers are never used).
    M, N, K = 8, 65536, 12288
    assert qg.workspace_size(qg.QG_OP_Q4_K, M, N, K) > (4 << 20)
    fake = 1 << 20
    rc = qg.lib().qgemv_q4_k_noalloc(C.c_void_p(fake), C.c_void_p(fake + (1 << 12)),
                                     C.c_void_p(fake + (1 << 13)), M, N, K,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == qg.QG_ERR_WORKSPACE
