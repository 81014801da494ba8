"""Seeded random tensors in the 16-bit storage formats of the workloads.

Every generator here is deterministic in (seed, flat element index): the flat
array is cut into fixed chunks of ``CHUNK`` elements and chunk ``c`` draws from
its own PCG64 stream ``SeedSequence(root, spawn_key=path + (c,))``, where
``seed`` is either an int ``root`` or a tuple ``(root, *path)`` (the path names
the tensor and the shard, so shards can be drawn independently).  The chunks are
filled in parallel threads (numpy releases the GIL while it fills), so the
values do not depend on the number of threads or on the machine.

Storage conventions shared by both consumers of these arrays:

* ``"f16"`` arrays are ``np.float16`` (IEEE binary16), rounded to nearest even
  from float32 by numpy.
* ``"bf16"`` arrays are ``np.uint16`` holding bfloat16 bit patterns, rounded to
  nearest even from float32 by :func:`f32_to_bf16_bits`.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "CHUNK", "DTYPES", "f32_to_bf16_bits", "bf16_bits_to_f32", "to_f32",
    "normal16", "uniform16", "integers16", "routing", "router_logits", "zipf_bias",
    "split_rows", "split_cols",
]

CHUNK = 1 << 22
DTYPES = ("f16", "bf16")


def _threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        n = os.cpu_count() or 1
    return max(1, min(n, 32))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f32(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Widen a stored 16-bit array to float32 (exact) for inspection in tests."""
    if dtype == "f16":
        return np.asarray(arr, dtype=np.float16).astype(np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(arr)
    raise ValueError(dtype)


def _store(src32: np.ndarray, dst: np.ndarray, dtype: str) -> None:
    if dtype == "f16":
        dst[...] = src32.astype(np.float16)
    else:
        dst[...] = f32_to_bf16_bits(src32)


def _seed_seq(seed, c: int) -> np.random.SeedSequence:
    """Seed of chunk ``c``: ``seed`` is an int or a tuple (root, *spawn path)."""
    if isinstance(seed, (tuple, list)):
        root, path = int(seed[0]), tuple(int(v) for v in seed[1:])
    else:
        root, path = int(seed), ()
    return np.random.SeedSequence(root, spawn_key=path + (c,))


def _chunked(seed, n: int, dtype: str, fill) -> np.ndarray:
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {DTYPES}, got {dtype!r}")
    out = np.empty(n, dtype=np.float16 if dtype == "f16" else np.uint16)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c: int) -> None:
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        g = np.random.Generator(np.random.PCG64(_seed_seq(seed, c)))
        _store(fill(g, hi - lo), out[lo:hi], dtype)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal16(seed, shape, std: float, dtype: str) -> np.ndarray:
    """N(0, std^2) samples (std is a standard deviation), stored as ``dtype``."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape, dtype=np.int64))
    s32 = np.float32(std)

    def fill(g, k):
        v = g.standard_normal(k, dtype=np.float32)
        if s32 != 1.0:
            v *= s32
        return v

    return _chunked(seed, n, dtype, fill).reshape(shape)


def uniform16(seed, shape, lo: float, hi: float, dtype: str) -> np.ndarray:
    """U[lo, hi) samples stored as ``dtype``."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape, dtype=np.int64))

    def fill(g, k):
        return g.uniform(lo, hi, k).astype(np.float32)

    return _chunked(seed, n, dtype, fill).reshape(shape)


def integers16(seed, shape, lo: int, hi: int, dtype: str) -> np.ndarray:
    """Integers drawn uniformly from [lo, hi] (inclusive), stored exactly as ``dtype``.

    Small integers are exact in both 16-bit formats, which makes every partial
    sum of a short dot product exact in fp32 as well.
    """
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape, dtype=np.int64))

    def fill(g, k):
        return g.integers(lo, hi + 1, k).astype(np.float32)

    return _chunked(seed, n, dtype, fill).reshape(shape)


def zipf_bias(E: int, s: float) -> np.ndarray:
    """Per-expert additive router bias ln(p_e) with p_e proportional to (e+1)^-s.

    Expert 0 is the most loaded; added to N(0, 1) router scores it skews a
    top-k gate toward a Zipf(s)-like load over the experts.
    """
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-float(s))
    p /= p.sum()
    return np.log(p)


def routing(seed, T: int, E: int, topk: int, zipf_s: float = 1.2,
            force_empty: tuple = ()):
    """Top-k routing of T tokens over E experts, drawn directly (no gate).

    Each token's topk distinct experts are drawn without replacement with
    probabilities proportional to (e+1)^-s, a Zipf(s) load with expert 0 the
    most loaded; experts listed in ``force_empty`` are never drawn (used to
    exercise empty experts).  The gate weights of a token are a flat Dirichlet
    draw over its k slots, largest in slot 0.  Router scores for the gate
    itself come from :func:`router_logits`.

    Returns ``(topk_ids int32 [T, topk], topk_weights float32 [T, topk])``.
    """
    empty = set(int(e) for e in force_empty)
    sel = np.array([e for e in range(E) if e not in empty], dtype=np.int64)
    if topk > sel.size:
        raise ValueError("topk larger than the number of selectable experts")
    g = np.random.Generator(np.random.PCG64(_seed_seq(seed, 0)))
    p = (sel + 1.0) ** (-float(zipf_s))
    p /= p.sum()
    ids = np.empty((T, topk), dtype=np.int32)
    for t in range(T):
        ids[t] = sel[g.choice(sel.size, size=topk, replace=False, p=p)]
    w = g.dirichlet(np.ones(topk), size=T) if T else np.zeros((0, topk))
    w = np.ascontiguousarray(np.sort(w, axis=1)[:, ::-1]).astype(np.float32)
    return ids, w


def router_logits(seed, T: int, E: int, zipf_s: float = 1.2, force_empty: tuple = ()):
    """Router scores float32 [T x E]: N(0, 1) plus the Zipf bias of :func:`zipf_bias`,
    -inf for the experts in ``force_empty``."""
    g = np.random.Generator(np.random.PCG64(_seed_seq(seed, 0)))
    L = (g.standard_normal((T, E)) + zipf_bias(E, zipf_s)[None, :]).astype(np.float32)
    for e in force_empty:
        L[:, int(e)] = -np.inf
    return L


def split_rows(a: np.ndarray, R: int):
    """R contiguous row blocks of ``a`` (rows must divide evenly)."""
    if a.shape[0] % R:
        raise ValueError("rows not divisible by R")
    h = a.shape[0] // R
    return [np.ascontiguousarray(a[r * h:(r + 1) * h]) for r in range(R)]


def split_cols(a: np.ndarray, R: int):
    """R contiguous column blocks of ``a`` (columns must divide evenly)."""
    if a.shape[-1] % R:
        raise ValueError("columns not divisible by R")
    w = a.shape[-1] // R
    return [np.ascontiguousarray(a[..., r * w:(r + 1) * w]) for r in range(R)]
