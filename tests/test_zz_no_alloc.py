"""GPU test of qgemv_q4_k_noalloc, the Q4_K GEMV for callers that cannot
allocate device memory (it takes its split-K scratch from a fixed array in the
library instead of a caller workspace).

Collected last on purpose: a run that stops at the first failure has run
every other test before this one. It also passes on its own in a fresh
process: it builds all its inputs itself and needs no state from other tests.
"""
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


@pytest.mark.parametrize("M", [16, 24, 32])
@pytest.mark.parametrize("N", [64, 256])
def test_noalloc_stays_on_cuda_cores_for_large_m(M, N):
    # From M = 16 up, qgemv_q4_k with a large enough workspace may take the
    # tensor-core prefill (error bound 2e-3 * sum |x w|). The no-alloc entry
    # point must keep the CUDA-core kernels and their f32 bound for every M,
    # whatever the size of its scratch array. x is 16-byte aligned here, which
    # the prefill also asks for.
    K = 4096
    qg.set_option(qg.QG_OPT_PREFILL_MIN_M, 16)
    c = synth.q4_k_case(3100 + M + N, N, K, M)
    w, x = to_dev(c["w"]), to_dev(c["x"])
    assert x.data_ptr() % 16 == 0
    for call in range(2):
        y = qg.qgemv_q4_k_noalloc(w, x, N=N)
        torch.cuda.synchronize()
        ref, bound = oracle.gemv_q4_k(c["w"], c["x"], M, N, K)
        assert_parity(y, ref, bound, what=f"no-alloc M={M} N={N} call {call}")
    assert qg.device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 3 slices x 8 rows x 65536 outputs x 4 bytes = 6 MiB > 4 MiB: refused with
    # QG_ERR_WORKSPACE before anything is enqueued. The buffers are real and
    # sized for the shape, so that a regression in the size check would run a
    # kernel on valid memory and show up as a wrong return code.
    M, N, K = 8, 65536, 12288
    assert qg.workspace_size(qg.QG_OP_Q4_K, M, N, K) > (4 << 20)
    w = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), dtype=torch.float32, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    rc = qg.lib().qgemv_q4_k_noalloc(w.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, K,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == qg.QG_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not y.any()
