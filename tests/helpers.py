"""Shared helpers for the GPU parity tests: device transfer and checks."""
import numpy as np
import torch

import oracle


def dev():
    return torch.device("cuda:0")


def to_dev(a, offset_bytes: int = 0):
    """numpy array -> CUDA tensor; with offset_bytes > 0 the data starts that
    many bytes into a larger uint8 buffer (to exercise unaligned pointers)."""
    a = np.ascontiguousarray(a)
    if offset_bytes == 0:
        return torch.from_numpy(a).to(dev())
    raw = a.view(np.uint8).ravel()
    buf = torch.zeros(raw.size + offset_bytes + 16, dtype=torch.uint8, device=dev())
    buf[offset_bytes:offset_bytes + raw.size] = torch.from_numpy(raw).to(dev())
    view = buf[offset_bytes:offset_bytes + raw.size]
    if a.dtype == np.uint8:
        return view
    raise ValueError("offset views are only made for uint8 data")


def assert_parity(y, ref, bound, rel=oracle.REL, abs_=oracle.ABS, what=""):
    yh = y.detach().cpu().numpy() if isinstance(y, torch.Tensor) else y
    ok, ratio = oracle.within(yh, ref, bound, rel, abs_)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} outputs outside tolerance, worst "
                             f"ratio {ratio:.3g}, first bad {idx.tolist()}")
    return ratio


def assert_bitwise(a, b, what=""):
    ah = a.detach().cpu().numpy() if isinstance(a, torch.Tensor) else a
    bh = b.detach().cpu().numpy() if isinstance(b, torch.Tensor) else b
    assert ah.shape == bh.shape, (what, ah.shape, bh.shape)
    eq = ah.view(np.uint32) == bh.view(np.uint32)
    if not eq.all():
        idx = np.argwhere(~eq)[:5]
        raise AssertionError(f"{what}: {int((~eq).sum())} words differ, first {idx.tolist()}")
