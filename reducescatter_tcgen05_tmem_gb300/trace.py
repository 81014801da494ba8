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


def summary(rec: dict) -> dict | None:
    """Where one traced call spent its time, from the records of the CTAs that
    issue their pair's MMAs (medians over those CTAs; shares of the call's
    span from the first producer start to the last epilogue end):
    k-loop (first operands in .. last commit of each unit), waits for the
    accumulator (last commit of the previous unit .. accumulator free) and for
    the first operands (accumulator free .. first operands in), and the idle
    time after the CTA's last unit.  None if nothing was recorded."""
    ok = rec["unit"] >= 0
    mma = np.any(rec["mma_end"] > 0, axis=1) & np.any(ok, axis=1)
    if not np.any(mma):
        return None
    t0 = rec["prod_start"][ok].min()
    t1 = rec["epi_end"][ok].max()
    span = float(t1 - t0)
    kl, wacc, wop, idle, items, it_k, it_e = [], [], [], [], [], [], []
    for b in np.nonzero(mma)[0]:
        it = np.nonzero(ok[b])[0]
        ma, mf, me = rec["mma_acc"][b, it], rec["mma_first"][b, it], rec["mma_end"][b, it]
        kl.append(np.sum(me - mf))
        wacc.append(np.sum(ma - np.concatenate([[t0], me[:-1]])))
        wop.append(np.sum(mf - ma))
        idle.append(t1 - me[-1])
        items.append(len(it))
        it_k.extend((me - mf).tolist())
        # (items whose partial stays in TMEM for the next rank of its group
        # have no epilogue of their own)
        ef, ee = rec["epi_full"][b, it], rec["epi_end"][b, it]
        it_e.extend((ee - ef)[ef > 0].tolist())
    med = lambda x: float(np.median(np.asarray(x, dtype=np.float64)))  # noqa: E731
    return {"span_us": round(span / 1e3, 1), "mma_ctas": int(np.sum(mma)), "units_per_cta": med(items),
            "kloop_share": round(med(kl) / span, 4), "acc_wait_share": round(med(wacc) / span, 4),
            "operand_wait_share": round(med(wop) / span, 4), "idle_after_last_share": round(med(idle) / span, 4),
            "unit_kloop_us": round(med(it_k) / 1e3, 2), "unit_epilogue_us": round(med(it_e) / 1e3, 2)}
