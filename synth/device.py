"""Copy a Problem's arrays to torch tensors (no arithmetic)."""
from __future__ import annotations

import numpy as np
import torch


def to_torch(p, device="cuda", pin: bool = False) -> dict:
    def t(a, dtype=None):
        if a is None:
            return None
        x = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            x = x.view(dtype)
        if device == "cpu":
            return x.pin_memory() if pin else x
        return x.to(device)

    return {"q": t(p.q), "dO": t(p.dO), "k": t(p.k), "v": t(p.v),
            "mask": t(p.mask.view(np.int16)) if p.mask is not None else None}
