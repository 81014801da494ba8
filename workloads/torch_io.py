"""Move generator arrays to and from torch tensors (bit-preserving views only)."""
from __future__ import annotations

import numpy as np


def to_device(arr: np.ndarray, dtype: str, device="cuda"):
    """A stored 16-bit array (np.float16 or bf16 bits as uint16) -> torch tensor."""
    import torch
    a = np.ascontiguousarray(arr)
    if dtype == "f16":
        t = torch.from_numpy(a.view(np.float16))
    elif dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        raise ValueError(dtype)
    return t.to(device)


def from_device(t) -> np.ndarray:
    """A 16-bit torch tensor -> np.float16 (fp16) or uint16 bit patterns (bf16)."""
    import torch
    c = t.detach().contiguous().cpu()
    if c.dtype == torch.float16:
        return c.numpy()
    if c.dtype == torch.bfloat16:
        return c.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(c.dtype)


def torch_dtype(dtype: str):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
