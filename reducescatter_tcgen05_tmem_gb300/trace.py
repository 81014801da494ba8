"""Decoding of the per-unit trace the fused kernels record (flux_opts_t.trace).

The kernel writes a header (grid size, records per CTA) and, for every work
item of every CTA, eight 64-bit words: a tag and seven %globaltimer stamps in
nanoseconds (see TraceField in the kernel header).  This module only reshapes
and names what the device wrote.
"""
from __future__ import annotations

import numpy as np

FIELDS = ("tag", "prod_start", "prod_end", "mma_acc", "mma_first", "mma_end", "epi_full", "epi_end")


def records(buf) -> dict:
    """Named arrays [grid, items] from a trace buffer (a torch tensor or numpy
    array of 64-bit words).  Empty records have tag 0; `unit` is the unit id
    (-1 for an empty record), `rank` the rank whose operands fed the item and
    `k0` its first k-slice."""
    if hasattr(buf, "detach"):
        buf = buf.detach().cpu().numpy()
    w = np.asarray(buf).view(np.uint64).ravel()
    grid, per = int(w[0]), int(w[1])
    rec = w[8:8 + grid * per * 8].reshape(grid, per, 8)
    out = {name: rec[:, :, i].astype(np.int64) for i, name in enumerate(FIELDS) if name != "tag"}
    tag = rec[:, :, 0]
    out["unit"] = (tag & 0xFFFFFFFF).astype(np.int64) - 1
    out["rank"] = ((tag >> 32) & 0xFF).astype(np.int64)
    out["k0"] = (tag >> 40).astype(np.int64)
    out["grid"], out["per_cta"] = grid, per
    return out
