"""Helpers shared by the GPU parity tests (no merge arithmetic here)."""
import numpy as np
import torch

GUARD = 36  # guard elements on each side of every output buffer (keeps 16-byte phase)
SENTINEL = -0x5A5A5A5B


def dev_i32(x: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).cuda()


def host(t) -> np.ndarray:
    return t.cpu().numpy()


def guarded_empty(total: int, offset_elems: int = 0):
    """An output view of `total` int32 with sentinel guard bands around it;
    `offset_elems` shifts the view's start by whole elements (misalignment)."""
    buf = torch.full((total + 2 * GUARD + 4,), SENTINEL, dtype=torch.int32, device="cuda")
    view = buf[GUARD + offset_elems: GUARD + offset_elems + total]
    return buf, view


def guards_intact(buf, total: int, offset_elems: int = 0) -> bool:
    h = host(buf)
    lo = h[: GUARD + offset_elems]
    hi = h[GUARD + offset_elems + total:]
    return bool(np.all(lo == SENTINEL) and np.all(hi == SENTINEL))


def shifted(t, offset_elems: int):
    """A copy of t whose data starts `offset_elems` int32 past a 16-byte boundary."""
    if offset_elems == 0:
        return t.clone()
    buf = torch.empty(t.numel() + 4, dtype=t.dtype, device=t.device)
    view = buf[offset_elems: offset_elems + t.numel()]
    view.copy_(t)
    return view
