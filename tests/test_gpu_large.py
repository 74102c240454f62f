"""GPU parity at the largest sizes the M <= 8 paths take: weight matrices of
2.4 to 2.7 GB (past 2^31 bytes, so every row offset needs 64-bit arithmetic), K at
the register-resident kernel's limit of 16384, and the concatenated row
list of a dual projection past 2^19 rows.

The weights are generated on the device (random codes, finite random block
scales), so the test needs no host copy of them; outputs are checked on
sampled rows (first, last, around the 2^31-byte boundary and random ones)
against the oracle run on those rows alone, at the f32 bar
|y - ref| <= 1e-5 * sum_k |x_k w_k| + 1e-6.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg

from helpers import assert_parity

pytestmark = pytest.mark.gpu

K = 16384
N = 1 << 18  # 2^18 rows of 9216 bytes: 2.4 GB per matrix


def _sample_rows(n_rows, row_bytes, seed):
    """First, last, the rows on both sides of byte 2^31, and random ones."""
    edge = (1 << 31) // row_bytes
    rng = np.random.default_rng(seed)
    rows = {0, 1, n_rows - 1, edge - 1, edge, edge + 1}
    rows |= set(int(r) for r in rng.integers(0, n_rows, 10))
    return sorted(r for r in rows if 0 <= r < n_rows)


def _random_blocks(n_rows, blocks, block_bytes, scale_bytes, gen):
    """Random code bytes with finite fp16 scales in the first scale_bytes of
    every block (values in [-0.02, 0.02))."""
    w = torch.randint(0, 256, (n_rows, blocks, block_bytes), dtype=torch.uint8, device="cuda",
                      generator=gen)
    nh = scale_bytes // 2
    d = (torch.rand((n_rows, blocks, nh), device="cuda", generator=gen) * 0.04 - 0.02).half()
    w[:, :, :scale_bytes] = d.view(torch.uint8).view(n_rows, blocks, scale_bytes)
    return w.view(n_rows, blocks * block_bytes)


@pytest.mark.parametrize("M", [1, 3])
def test_q4_0_dual_2_4_gb_per_weight(M):
    gen = torch.Generator(device="cuda").manual_seed(11 + M)
    wa = _random_blocks(N, K // 32, 18, 2, gen)
    wb = _random_blocks(N, K // 32, 18, 2, gen)
    row_bytes = wa.shape[1]
    assert N * row_bytes > (1 << 31)
    x = torch.randn((M, K), device="cuda", generator=gen)
    ya, yb = qg.qgemv_dual_q4_0(wa, wb, x, N=N)
    torch.cuda.synchronize()
    rows = _sample_rows(N, row_bytes, 100 + M)
    xh = x.cpu().numpy()
    for w, y, name in ((wa, ya, "y_a"), (wb, yb, "y_b")):
        wr = w[rows].cpu().numpy()
        ref, bound = oracle.gemv_q4_0(wr, xh, M, len(rows), K)
        assert_parity(y[:, rows].cpu().numpy(), ref, bound, what=f"q4_0 dual {name} M={M}")
    del wa, wb
    torch.cuda.empty_cache()


def test_q4_k_2_4_gb():
    gen = torch.Generator(device="cuda").manual_seed(21)
    # 144-byte super-blocks: d and dmin (fp16) first, then scales and nibbles.
    w = _random_blocks(N, K // 256, 144, 4, gen)
    row_bytes = w.shape[1]
    assert N * row_bytes > (1 << 31)
    x = torch.randn((1, K), device="cuda", generator=gen)
    y = qg.qgemv_q4_k(w, x, N=N)
    torch.cuda.synchronize()
    rows = _sample_rows(N, row_bytes, 200)
    ref, bound = oracle.gemv_q4_k(w[rows].cpu().numpy(), x.cpu().numpy(), 1, len(rows), K)
    assert_parity(y[:, rows].cpu().numpy(), ref, bound, what="q4_k 2.4 GB")
    del w
    torch.cuda.empty_cache()


def test_affine_u8_2_7_gb():
    gen = torch.Generator(device="cuda").manual_seed(31)
    n, gs = (1 << 17) + (1 << 15), 64  # 2.7 GB of codes
    q = torch.randint(0, 256, (n, K), dtype=torch.uint8, device="cuda", generator=gen)
    s = torch.rand((n, K // gs), device="cuda", generator=gen) * 0.009 + 0.001
    b = torch.rand((n, K // gs), device="cuda", generator=gen) * -0.08
    x = torch.randn((1, K), device="cuda", generator=gen)
    y = qg.qmm_affine(x, q, s, b, gs, 0)
    torch.cuda.synchronize()
    rows = _sample_rows(n, K, 300)
    ref, bound = oracle.qmm_affine(x.cpu().numpy(), q[rows].cpu().numpy(), s[rows].cpu().numpy(),
                                   b[rows].cpu().numpy(), 1, len(rows), K, gs, False)
    assert_parity(y[:, rows].cpu().numpy(), ref, bound, what="affine u8 2.7 GB")
    del q
    torch.cuda.empty_cache()
