"""Shared parity helpers for the GPU tests (tolerance of the path's statement)."""
import numpy as np

# floating point bar: relative Frobenius error <= 5e-3 and every element within
# 1e-2 * max|ref| of the float64 oracle
REL_FROB = 5e-3
ELEM_FRAC = 1e-2


def check_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if ref.size == 0:
        return
    scale = float(np.max(np.abs(ref)))
    err = np.abs(got - ref)
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / denom if denom > 0 else float(np.linalg.norm(got - ref))
    worst = float(err.max())
    assert rel <= REL_FROB, f"{what}: relative Frobenius error {rel:.3e} > {REL_FROB}"
    assert worst <= ELEM_FRAC * max(scale, 1e-30), \
        f"{what}: max |err| {worst:.3e} > {ELEM_FRAC} * max|ref| ({scale:.3e})"
    return rel, worst
