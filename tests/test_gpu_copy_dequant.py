"""GPU parity: QKV split and the dequantization exports, bit-exact against
the oracle (the only correct answers for a copy and for a dequantization)."""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemv_dequant_gb300 as qg
from bit_quantized_gemv_dequant_gb300 import synth

from helpers import assert_bitwise, dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seq,qs,ks,vs", [(1, 4, 4, 4), (7, 8, 4, 12), (33, 5, 3, 9),
                                          (3, 1, 1, 1), (64, 256, 256, 512)])
def test_qkv_split_bitwise(seq, qs, ks, vs):
    x = synth.qkv_case(100 + seq, seq, qs, ks, vs)
    bits = x.view(np.uint32)
    bits[0, 0] = 0x7FC00123  # NaN payloads must survive
    bits[-1, -1] = 0xFF800001
    q, k, v = qg.qkv_split(to_dev(x), qs, ks, vs)
    oq, ok_, ov = oracle.qkv_split(x, seq, qs, ks, vs)
    assert_bitwise(q, oq, "q")
    assert_bitwise(k, ok_, "k")
    assert_bitwise(v, ov, "v")


def test_qkv_split_full_config():
    seq, qs, ks, vs = 4096, 2048, 2048, 4096
    x = synth.qkv_case(4, seq, qs, ks, vs)
    q, k, v = qg.qkv_split(to_dev(x), qs, ks, vs)
    oq, ok_, ov = oracle.qkv_split(x, seq, qs, ks, vs)
    assert_bitwise(q, oq, "q")
    assert_bitwise(k, ok_, "k")
    assert_bitwise(v, ov, "v")


def test_qkv_split_unaligned_pointer_path():
    seq, qs, ks, vs = 9, 6, 2, 10
    x = synth.qkv_case(7, seq, qs, ks, vs)
    big = torch.zeros(x.size + 1, dtype=torch.float32, device=dev())
    big[1:] = torch.from_numpy(x.ravel()).to(dev())
    src = big[1:].view(seq, qs + ks + vs)  # 4-byte but not 16-byte aligned
    q, k, v = qg.qkv_split(src, qs, ks, vs)
    oq, ok_, ov = oracle.qkv_split(x, seq, qs, ks, vs)
    assert_bitwise(q, oq, "q")
    assert_bitwise(k, ok_, "k")
    assert_bitwise(v, ov, "v")


@pytest.mark.parametrize("N,K", [(1, 32), (5, 96), (37, 1024), (64, 4096)])
def test_dequant_q4_0_bitexact(N, K):
    case = synth.q4_0_case(200 + N, N, K, 1)
    out = qg.dequant_q4_0(to_dev(case["w"]), N, K)
    assert_bitwise(out, oracle.dequant_q4_0(case["w"], N, K), "dequant_q4_0")


def test_dequant_q4_0_golden_edge_blocks():
    import json, os
    from conftest import GOLDEN
    with open(os.path.join(GOLDEN, "q4_0_blocks.json")) as f:
        fx = json.load(f)
    raw = np.concatenate([np.frombuffer(bytes.fromhex(b["hex"]), dtype=np.uint8)
                          for b in fx["blocks"]])
    n = len(fx["blocks"])
    out = qg.dequant_q4_0(to_dev(raw), 1, 32 * n)
    exp = np.array(sum((b["expected"] for b in fx["blocks"]), []), dtype=np.float32)[None, :]
    assert_bitwise(out, exp, "golden Q4_0 blocks")


@pytest.mark.parametrize("N,K", [(1, 256), (3, 512), (33, 4096)])
def test_dequant_q4_k_bitexact(N, K):
    case = synth.q4_k_case(300 + N, N, K, 1)
    out = qg.dequant_q4_k(to_dev(case["w"]), N, K)
    assert_bitwise(out, oracle.dequant_q4_k(case["w"], N, K), "dequant_q4_k")


def test_dequant_q4_k_random_bytes():
    # Arbitrary bytes with finite fp16 headers: every 6-bit pair and nibble.
    rng = np.random.default_rng(9)
    N, K = 16, 1024
    w = rng.integers(0, 256, size=(N, K // 256, 144), dtype=np.uint8)
    w[..., 1] &= 0x3B  # keep d, dmin finite
    w[..., 3] &= 0x3B
    w = w.reshape(N, -1)
    out = qg.dequant_q4_k(to_dev(w), N, K)
    assert_bitwise(out, oracle.dequant_q4_k(w, N, K), "dequant_q4_k random")


@pytest.mark.parametrize("packed", [0, 1])
@pytest.mark.parametrize("N,K,gs", [(4, 64, 64), (9, 256, 2), (17, 512, 128), (8, 4096, 64)])
def test_dequant_affine_bitexact(N, K, gs, packed):
    case = synth.affine_case(400 + N, N, K, 1, gs)
    q = case["q_packed"] if packed else case["q"]
    out = qg.dequant_affine(to_dev(q), to_dev(case["s"]), to_dev(case["b"]), N, K, gs, packed)
    exp = oracle.dequant_affine(q, case["s"], case["b"], N, K, gs, packed)
    assert_bitwise(out, exp, "dequant_affine")
