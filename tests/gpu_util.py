"""Shared set-up for the GPU parity tests: build once, move synthetic inputs
to the device in the dtype the library computes in."""
import numpy as np
import torch

import __graft_entry__

_BUILT = False


def device():
    global _BUILT
    if not _BUILT:
        __graft_entry__.build()
        _BUILT = True
    return torch.device("cuda:0")


def to_dev(a: np.ndarray, dtype: str):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)   # values are already bf16: exact
    elif dtype == "f32":
        t = t.to(torch.float32)
    elif dtype == "i32":
        t = t.to(torch.int32)
    return t.to(device())
