"""GPU parity of qgemv_dual_q4_0_host: the dual Q4_0 projection with x, y_a
and y_b in host memory, returning once the outputs hold the result.

Both routes are covered: page-locked buffers with M <= 2 (x fetched into the
workspace by a kernel, the outputs stored by the GEMV straight into host
memory) and pageable buffers or M >= 3 (one copy per buffer through the
workspace). Each result is compared bit for bit with qgemv_dual_q4_0 on
device copies of the same inputs, and with the oracle's f64 reference under
the f32 GEMV bound |y - ref| <= 1e-5 * sum_k |x_k w_k| + 1e-6. Also covered:
the full workload size under every QG_OPT_PDL mode with fresh x every call
(the zero-copy GEMV waits for its fetch even when calls are declared
independent), which route ran (the zero-copy route leaves the workspace's
output staging untouched), a pinned x that is not 16-byte aligned, and the
argument checks.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, assert_parity, to_dev

pytestmark = pytest.mark.gpu


def host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t.clone()


def round256(v):
    return (v + 255) // 256 * 256


@pytest.fixture
def pdl_mode():
    old = qg.get_option(qg.QG_OPT_PDL)
    yield
    qg.set_option(qg.QG_OPT_PDL, old)


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("M", [1, 2, 3, 8])
@pytest.mark.parametrize("N,K", [(37, 256), (300, 4096), (23, 12288)])
def test_host_call_matches_device_call(pinned, M, N, K):
    c = synth.q4_0_case(7100 + M + N, N, K, M, dual=True)
    wa, wb = to_dev(c["w"]), to_dev(c["w_b"])
    ha, hb = qg.qgemv_dual_q4_0_host(wa, wb, host(c["x"], pinned), N=N)
    assert ha.device.type == "cpu" and hb.device.type == "cpu"
    da, db = qg.qgemv_dual_q4_0(wa, wb, to_dev(c["x"]), N=N)
    assert_bitwise(ha, da, f"host vs device y_a M={M} N={N} K={K} pinned={pinned}")
    assert_bitwise(hb, db, f"host vs device y_b M={M} N={N} K={K} pinned={pinned}")
    (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], c["x"], M, N, K)
    assert_parity(ha, ra, ba, what=f"host y_a M={M} N={N} K={K}")
    assert_parity(hb, rb, bb, what=f"host y_b M={M} N={N} K={K}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_host_full_workload_fresh_x_every_call(mode, pdl_mode):
    """N = K = 4096, M = 1, page-locked buffers: three calls in a row, x
    rewritten on the host before each; every result matches the oracle for
    the x of its own call."""
    qg.set_option(qg.QG_OPT_PDL, mode)
    N = K = 4096
    c = synth.q4_0_case(1, N, K, 1, dual=True)
    wa, wb = to_dev(c["w"]), to_dev(c["w_b"])
    x = torch.empty((1, K), dtype=torch.float32).pin_memory()
    ya = torch.empty((1, N), dtype=torch.float32).pin_memory()
    yb = torch.empty((1, N), dtype=torch.float32).pin_memory()
    rng = np.random.default_rng(mode)
    for i in range(3):
        xi = c["x"] if i == 0 else rng.standard_normal((1, K)).astype(np.float32)
        x.copy_(torch.from_numpy(xi))
        qg.qgemv_dual_q4_0_host(wa, wb, x, ya, yb, N=N)
        (ra, ba), (rb, bb) = oracle.gemv_dual_q4_0(c["w"], c["w_b"], xi, 1, N, K)
        assert_parity(ya, ra, ba, what=f"PDL {mode} call {i} y_a")
        assert_parity(yb, rb, bb, what=f"PDL {mode} call {i} y_b")


@pytest.mark.parametrize("pinned,M,direct", [(True, 1, True), (True, 2, True),
                                             (True, 3, False), (False, 1, False)])
def test_host_route_taken(pinned, M, direct):
    """The zero-copy route never touches the output staging at the end of
    the workspace; the copy route leaves y_a there."""
    N, K = 96, 1024
    c = synth.q4_0_case(7200 + M, N, K, M, dual=True)
    wa, wb = to_dev(c["w"]), to_dev(c["w_b"])
    need = qg.workspace_size(qg.QG_OP_DUAL_Q4_0_HOST, M, N, K)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    ya, yb = qg.qgemv_dual_q4_0_host(wa, wb, host(c["x"], pinned), N=N, workspace=ws)
    stage = round256(4 * M * K) + 2 * round256(4 * M * N)
    off = (need - stage) // 256 * 256 + round256(4 * M * K)
    staged_a = ws[off:off + 4 * M * N].cpu().numpy()
    if direct:
        assert (staged_a == 0xFF).all(), "zero-copy route wrote the output staging"
    else:
        assert_bitwise(staged_a.view(np.float32).reshape(M, N), ya, "staged y_a")
    da, _ = qg.qgemv_dual_q4_0(wa, wb, to_dev(c["x"]), N=N)
    assert_bitwise(ya, da, "host vs device y_a")


def test_host_misaligned_pinned_x_takes_copies():
    """A page-locked x 4 bytes off a 16-byte boundary is staged by a copy
    (the fetch kernel moves 16-byte vectors); results stay bitwise equal."""
    M, N, K = 1, 200, 2048
    c = synth.q4_0_case(7300, N, K, M, dual=True)
    wa, wb = to_dev(c["w"]), to_dev(c["w_b"])
    buf = torch.empty(M * K + 4, dtype=torch.float32).pin_memory()
    x = buf[1:1 + M * K].view(M, K)
    assert x.data_ptr() % 16 == 4
    x.copy_(torch.from_numpy(c["x"]))
    ya, yb = qg.qgemv_dual_q4_0_host(wa, wb, x, N=N)
    da, db = qg.qgemv_dual_q4_0(wa, wb, to_dev(c["x"]), N=N)
    assert_bitwise(ya, da, "misaligned pinned x y_a")
    assert_bitwise(yb, db, "misaligned pinned x y_b")


def test_host_argument_checks():
    M, N, K = 1, 64, 256
    c = synth.q4_0_case(7400, N, K, M, dual=True)
    wa, wb = to_dev(c["w"]), to_dev(c["w_b"])
    x = host(c["x"], True)
    ya = torch.empty((M, N), dtype=torch.float32).pin_memory()
    yb = torch.empty((M, N), dtype=torch.float32).pin_memory()
    L = qg.lib()
    st = torch.cuda.current_stream().cuda_stream
    need = qg.workspace_size(qg.QG_OP_DUAL_Q4_0_HOST, M, N, K)
    assert need >= 4 * M * K + 2 * 4 * M * N
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (wa.data_ptr(), wb.data_ptr(), x.data_ptr(), ya.data_ptr(), yb.data_ptr(), M, N, K)
    # No workspace, or one byte short of the staging: refused before anything
    # runs.
    stage = round256(4 * M * K) + 2 * round256(4 * M * N)
    assert L.qgemv_dual_q4_0_host(*args, None, 0, st) == qg.QG_ERR_WORKSPACE
    assert L.qgemv_dual_q4_0_host(*args, ws.data_ptr(), stage - 1, st) == qg.QG_ERR_WORKSPACE
    assert L.qgemv_dual_q4_0_host(*args, ws.data_ptr(), need, st) == qg.QG_OK
    # y_a on top of x, y_b on top of y_a.
    bad = (wa.data_ptr(), wb.data_ptr(), x.data_ptr(), x.data_ptr(), yb.data_ptr(), M, N, K)
    assert L.qgemv_dual_q4_0_host(*bad, ws.data_ptr(), need, st) == qg.QG_ERR_INVALID_ARG
    bad = (wa.data_ptr(), wb.data_ptr(), x.data_ptr(), ya.data_ptr(), ya.data_ptr(), M, N, K)
    assert L.qgemv_dual_q4_0_host(*bad, ws.data_ptr(), need, st) == qg.QG_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        qg.qgemv_dual_q4_0_host(wa, wb, to_dev(c["x"]), N=N)
