"""Plain, slow, obviously correct CPU oracle (numpy, float64).

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Nothing in the CUDA
path imports this module; it shares no code, table or constant with it.

What it computes and where that is defined
------------------------------------------
* The dense tensor-parallel MLP of the FLUX paper (FLUX paper review,
  section "三、技术架构 / MLP 前向传播"):
      Output1 = GEMM(AllGather(X), W1)                       -> :func:`ag_gemm`
      Output2 = ReduceScatter(GEMM(Output1, W2))             -> :func:`gemm_rs`
  The shard directions follow the Megatron-style reading: X is split by rows
  (tokens) and W1 [K x N] by columns; Output1 is split by columns and W2 by
  rows, so rank r's partial product A_r . B_r covers its K/R slice and owner
  rank o receives rows [o M/R, (o+1) M/R) of the sum over ranks.
* The COMET MoE variant (Comet article, section "COMET 的技术原理": the
  shared tensor is decomposed along the token dimension, tokens are gathered
  to experts, and the expert outputs are combined back by token):
      routing (stable counting sort of the top-k slots by expert) -> :func:`moe_route`
      layer0 = gather-by-expert(AllGather(X)) . W1_{e,r}         -> :func:`moe_layer0`
      layer1 = ReduceScatter_by_token(sum_k g_k . (H_r . W2_{e,r})) -> :func:`moe_layer1`
  the same two layers under the EP x TP split of the experts (the EP/TP ratio
  of that section) -> :func:`moe_ep_layer0`, :func:`moe_ep_layer1`, and the
  top-k gate that produces the routing from router scores -> :func:`moe_topk_gate`.

Precision: the pages fix none, so every floating-point result here is the
exact float64 value of the stored 16-bit inputs combined in float64 (a
library matmul serves as the dot-product step).  Ranks are summed in
ascending rank order and top-k contributions in ascending k, as the plain
reading of "sum over ranks" states.  Routing is integer and exact.

Storage formats of the inputs: "f16" arrays are np.float16; "bf16" arrays are
np.uint16 bfloat16 bit patterns, which :func:`widen` decodes itself.

Every function here is pinned by ``tests/test_oracle.py`` to facts other
than its own formula (brute force on tiny inputs, identities, closed forms,
library special cases).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "widen", "round_to", "gemm", "ag_gemm", "gemm_rs", "moe_route",
    "moe_layer0", "moe_layer1", "ag_gemm_at", "gemm_rs_at", "moe_layer0_rows",
    "moe_layer1_rows", "moe_ep_layer0", "moe_ep_layer1", "moe_ep_layer1_rows", "moe_topk_gate",
]


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def widen(a, dtype: str) -> np.ndarray:
    """Exact float64 value of a stored 16-bit array.

    bf16 is the upper half of an IEEE binary32, so its value is the float32
    whose high 16 bits are the stored pattern and whose low 16 bits are zero.
    """
    if dtype == "f16":
        return np.asarray(a, dtype=np.float16).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype in ("f32", "f64"):
        return np.asarray(a, dtype=np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the 16-bit storage format, nearest-even.

    Returns the rounded values as float64.  fp16 uses numpy's correctly
    rounded double->half conversion.  bf16 keeps 8 significant bits: the
    significand from frexp (in [0.5, 1)) is scaled by 2^8 and rounded
    half-to-even by rint.  (Normal range only; the workloads never reach the
    bf16 subnormal range.)
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        m, e = np.frexp(x)
        return np.ldexp(np.rint(m * 256.0) / 256.0, e)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# dense GEMM and the two fused collectives
# --------------------------------------------------------------------------
def gemm(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """C[i, j] = sum_k A[i, k] B[k, j] in float64 (the non-split GEMM)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"bad GEMM shapes {A.shape} x {B.shape}")
    return A @ B


def ag_gemm(x_shards, w_shards, dtype: str):
    """Output1_r = GEMM(AllGather(X), W1_r) for every rank r.

    AllGather concatenates the row shards X_0 .. X_{R-1} in rank order
    (FLUX paper review, "MLP 前向传播", first GEMM).  Returns R float64 arrays
    of shape [M, N/R].
    """
    R = len(x_shards)
    if len(w_shards) != R or R == 0:
        raise ValueError("need R x shards and R w shards")
    xfull = np.concatenate([widen(x, dtype) for x in x_shards], axis=0)
    return [gemm(xfull, widen(w, dtype)) for w in w_shards]


def gemm_rs(a_shards, b_shards, dtype: str):
    """Output2_o = rows [o M/R, (o+1) M/R) of sum_r GEMM(A_r, B_r).

    Rank r's partial is A_r . B_r over its K/R slice; the partials are summed
    in ascending rank order, then scattered so that owner o keeps its row chunk
    (FLUX paper review, "MLP 前向传播", second GEMM).  Returns R float64 arrays
    of shape [M/R, N].
    """
    R = len(a_shards)
    if len(b_shards) != R or R == 0:
        raise ValueError("need R a shards and R b shards")
    M = np.asarray(a_shards[0]).shape[0]
    if M % R:
        raise ValueError("M must divide by R")
    total = None
    for r in range(R):
        p = gemm(widen(a_shards[r], dtype), widen(b_shards[r], dtype))
        total = p if total is None else total + p
    h = M // R
    return [total[o * h:(o + 1) * h].copy() for o in range(R)]


def ag_gemm_at(x_shards, w_shards, dtype: str, r: int, rows, cols) -> np.ndarray:
    """Output1_r[rows[i], cols[i]] for sampled index pairs (float64): the dot
    product of gathered row rows[i] of X with column cols[i] of W1_r (only the
    sampled columns of W1_r are widened)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    m_local = np.asarray(x_shards[0]).shape[0]
    out = np.empty(rows.shape[0], dtype=np.float64)
    ucols, cidx = np.unique(cols, return_inverse=True)
    w = widen(np.asarray(w_shards[r])[:, ucols], dtype)  # [K x sampled columns]
    xrows = {}
    for i, (row, ci) in enumerate(zip(rows, cidx)):
        if int(row) not in xrows:
            s, lr = divmod(int(row), m_local)
            xrows[int(row)] = widen(np.asarray(x_shards[s])[lr], dtype)
        out[i] = float(np.dot(xrows[int(row)], w[:, ci]))
    return out


def gemm_rs_at(a_shards, b_shards, dtype: str, o: int, rows, cols) -> np.ndarray:
    """Output2_o[rows[i], cols[i]] (rows local to owner o) for sampled pairs:
    sum over ranks r ascending of the dot product of row o M/R + rows[i] of A_r
    with column cols[i] of B_r (only the sampled rows and columns are widened)."""
    R = len(a_shards)
    M = np.asarray(a_shards[0]).shape[0]
    h = M // R
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    urows, ridx = np.unique(rows, return_inverse=True)
    ucols, cidx = np.unique(cols, return_inverse=True)
    a = [widen(np.asarray(a_shards[r])[o * h + urows], dtype) for r in range(R)]
    b = [widen(np.asarray(b_shards[r])[:, ucols], dtype) for r in range(R)]
    out = np.zeros(rows.shape[0], dtype=np.float64)
    for i, (ri, ci) in enumerate(zip(ridx, cidx)):
        acc = 0.0
        for r in range(R):
            acc = acc + float(np.dot(a[r][ri], b[r][:, ci]))
        out[i] = acc
    return out


# --------------------------------------------------------------------------
# MoE
# --------------------------------------------------------------------------
def moe_route(topk_ids: np.ndarray, E: int):
    """Stable counting sort of the top-k slots by expert.

    Slot s = t * topk + k holds expert id[t, k].  Returns int32 arrays
      counts[e]       number of slots routed to expert e
      offsets[e]      exclusive prefix sum of counts (offsets[E] = T * topk)
      slot_to_row[s]  offsets[id[s]] + (number of earlier slots with the same id)
      row_to_slot[r]  the inverse permutation
    i.e. rows are grouped by expert in ascending expert order and, within one
    expert, keep ascending slot order (tokens gathered to experts, Comet
    article, "共享张量依赖解析").
    """
    ids = np.asarray(topk_ids).reshape(-1)
    n = ids.shape[0]
    counts = [0] * E
    for s in range(n):
        e = int(ids[s])
        if e < 0 or e >= E:
            raise ValueError(f"expert id {e} out of range [0, {E})")
        counts[e] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    seen = [0] * E
    slot_to_row = [0] * n
    row_to_slot = [0] * n
    for s in range(n):
        e = int(ids[s])
        row = offsets[e] + seen[e]
        seen[e] += 1
        slot_to_row[s] = row
        row_to_slot[row] = s
    i32 = lambda v: np.asarray(v, dtype=np.int32)  # noqa: E731
    return i32(counts), i32(offsets), i32(slot_to_row), i32(row_to_slot)


def moe_topk_gate(logits, topk: int):
    """Top-k expert choice and gate weights of each token from its router scores.

    The pages name the MoE layer (COMET article, "COMET 是什么") but not its
    gate; reading: the plainest Mixture-of-Experts gate.  For token t with fp32
    scores s[t, 0..E-1] (a NaN counts as -inf):
      ids[t]  the topk experts with the largest scores, largest first, equal
              scores in ascending expert order;
      w[t, j] = exp(s_j - s_0) / sum_i exp(s_i - s_0) over the chosen scores
              (s_0 the largest), i.e. softmax over all E renormalised over the
              chosen k.  If s_0 is infinite the chosen scores equal to s_0
              share the weight equally and the others get 0 (the limit).
    Returns (int32 [T, topk], float64 [T, topk]).  Decisions are taken on the
    fp32 values exactly; the weights are float64.
    """
    import math
    L = np.asarray(logits, dtype=np.float32)
    T, E = L.shape
    if not 1 <= topk <= E:
        raise ValueError("need 1 <= topk <= E")
    ids = np.zeros((T, topk), dtype=np.int32)
    w = np.zeros((T, topk), dtype=np.float64)
    for t in range(T):
        s = [float("-inf") if math.isnan(float(v)) else float(v) for v in L[t]]
        chosen = sorted(range(E), key=lambda e: (-s[e], e))[:topk]
        top = s[chosen[0]]
        if math.isinf(top):
            z = [1.0 if s[e] == top else 0.0 for e in chosen]
        else:
            z = [math.exp(s[e] - top) for e in chosen]
        total = math.fsum(z)
        ids[t] = chosen
        w[t] = [v / total for v in z]
    return ids, w


def moe_layer0(x_shards, w1_shards, topk_ids, E: int, dtype: str):
    """layer0: H_r[row] = AllGather(X)[token(row)] . W1_r[expert(row)].

    Rows are in the grouped (expert-sorted) order of :func:`moe_route`; for row
    ``row`` the slot is s = row_to_slot[row], the token t = s // topk and the
    expert id[t, s % topk].  Returns (list of R float64 [T*topk, F/R],
    routing tuple).
    """
    ids = np.asarray(topk_ids)
    T, topk = ids.shape
    routing_ = moe_route(ids, E)
    counts, offsets, slot_to_row, row_to_slot = routing_
    xfull = np.concatenate([widen(x, dtype) for x in x_shards], axis=0)
    if xfull.shape[0] != T:
        raise ValueError("token count mismatch")
    outs = []
    for w1 in w1_shards:
        w = widen(w1, dtype)  # [E, H, F/R]
        h = np.zeros((T * topk, w.shape[2]), dtype=np.float64)
        for e in range(E):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            if hi == lo:
                continue
            tokens = row_to_slot[lo:hi].astype(np.int64) // topk
            h[lo:hi] = gemm(xfull[tokens], w[e])
        outs.append(h)
    return outs, routing_


def moe_layer1(h_shards, w2_shards, topk_ids, topk_weights, E: int, dtype: str,
               routing_=None, h_dtype: str | None = None):
    """layer1: Y[t] = sum_r sum_k g[t,k] (H_r[row(t,k)] . W2_r[id[t,k]]), scattered by token.

    Rank order ascending, then k ascending.  Owner o receives token rows
    [o T/R, (o+1) T/R).  ``h_dtype`` is the storage format of the H shards
    ("f64" when chaining exact layer0 values; defaults to ``dtype``).
    Returns R float64 arrays [T/R, H].
    """
    ids = np.asarray(topk_ids)
    g = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    T, topk = ids.shape
    R = len(h_shards)
    if T % R:
        raise ValueError("T must divide by R")
    if routing_ is None:
        routing_ = moe_route(ids, E)
    _, offsets, slot_to_row, row_to_slot = routing_
    hd = dtype if h_dtype is None else h_dtype
    Y = None
    s2r = np.asarray(slot_to_row, dtype=np.int64).reshape(T, topk)
    for r in range(R):
        hr = widen(h_shards[r], hd)
        w = widen(w2_shards[r], dtype)  # [E, F/R, H]
        P = np.zeros((T * topk, w.shape[2]), dtype=np.float64)
        for e in range(E):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            if hi > lo:
                P[lo:hi] = gemm(hr[lo:hi], w[e])
        if Y is None:
            Y = np.zeros((T, w.shape[2]), dtype=np.float64)
        for k in range(topk):
            # contribution of slot (t, k) of rank r, for every token t at once
            Y = Y + g[:, k:k + 1] * P[s2r[:, k]]
    h = T // R
    return [Y[o * h:(o + 1) * h].copy() for o in range(R)]


def moe_ep_layer0(x_shards, w1_ep, topk_ids, E: int, dtype: str, tp: int = 1):
    """Expert-parallel layer0: H[row] = X[token(row)] . W1_e, e the row's expert.

    The expert-parallel layout of the MoE layer (COMET article, "COMET 的技术
    原理", its EP x TP ratio).  The R = len(w1_ep) ranks form EP = R / tp
    groups of tp ranks; group g holds experts [g E/EP, (g+1) E/EP), and rank
    r = g tp + t of the group holds column block t (F/tp wide) of each:
    ``w1_ep[r][e - g E/EP]`` is [H, F/tp].  tp = 1 is pure expert parallel
    (whole experts per rank), tp = R the tensor-parallel layout of
    :func:`moe_layer0`.  The dispatch sends each routed token row to the ranks
    of its expert; rows keep the grouped order of :func:`moe_route`, so group
    g's rows are [offsets[g E/EP], offsets[(g+1) E/EP]).  Returns (float64
    [T*topk, F] with rank r's block at those rows and columns
    [t F/tp, (t+1) F/tp), routing tuple).
    """
    ids = np.asarray(topk_ids)
    T, topk = ids.shape
    R = len(w1_ep)
    if tp < 1 or R % tp:
        raise ValueError("tp must divide R")
    ep = R // tp
    if E % ep:
        raise ValueError("E must divide by R / tp")
    el = E // ep
    routing_ = moe_route(ids, E)
    _, offsets, _, row_to_slot = routing_
    xfull = np.concatenate([widen(x, dtype) for x in x_shards], axis=0)
    if xfull.shape[0] != T:
        raise ValueError("token count mismatch")
    fb = np.asarray(w1_ep[0]).shape[2]  # F / tp
    h = np.zeros((T * topk, fb * tp), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        tokens = row_to_slot[lo:hi].astype(np.int64) // topk
        g = e // el
        for t in range(tp):
            w = widen(np.asarray(w1_ep[g * tp + t])[e % el], dtype)  # [H, F/tp]
            h[lo:hi, t * fb:(t + 1) * fb] = gemm(xfull[tokens], w)
    return h, routing_


def moe_ep_layer1(h, w2_ep, topk_ids, topk_weights, E: int, dtype: str, R: int,
                  routing_=None, h_dtype: str | None = None, tp: int = 1):
    """Expert-parallel layer1 and combine: Y[t] = sum_k g[t,k] (H[row(t,k)] . W2_{id[t,k]}).

    Layout as in :func:`moe_ep_layer0`: rank r = g tp + t holds row block t
    (F/tp tall) of each expert of group g, ``w2_ep[r][e - g E/EP]`` [F/tp, H],
    and multiplies it with the matching column block of H.  A (token, k)
    slot sums its tp partials (t ascending), the slots are weighted and added
    k ascending, and the combine returns every token row to its owner: owner
    o receives rows [o T/R, (o+1) T/R).  Returns R float64 arrays [T/R, H].
    """
    ids = np.asarray(topk_ids)
    g = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    T, topk = ids.shape
    if tp < 1 or R % tp or len(w2_ep) != R:
        raise ValueError("tp must divide R, one w2 block per rank")
    ep = R // tp
    if T % R or E % ep:
        raise ValueError("T must divide by R and E by R / tp")
    el = E // ep
    if routing_ is None:
        routing_ = moe_route(ids, E)
    _, offsets, slot_to_row, _ = routing_
    hd = dtype if h_dtype is None else h_dtype
    hh = widen(h, hd)
    fb = np.asarray(w2_ep[0]).shape[1]  # F / tp
    Hn = np.asarray(w2_ep[0]).shape[2]
    P = np.zeros((T * topk, Hn), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        grp = e // el
        for t in range(tp):
            w = widen(np.asarray(w2_ep[grp * tp + t])[e % el], dtype)
            P[lo:hi] = P[lo:hi] + gemm(hh[lo:hi, t * fb:(t + 1) * fb], w)
    s2r = np.asarray(slot_to_row, dtype=np.int64).reshape(T, topk)
    Y = np.zeros((T, Hn), dtype=np.float64)
    for k in range(topk):
        Y = Y + g[:, k:k + 1] * P[s2r[:, k]]
    n = T // R
    return [Y[o * n:(o + 1) * n].copy() for o in range(R)]


def moe_layer0_rows(x_shards, w1_shards, topk_ids, E: int, dtype: str, r: int, rows):
    """H_r[rows] (full F/R width) for sampled grouped-order rows (float64)."""
    ids = np.asarray(topk_ids)
    T, topk = ids.shape
    _, _, _, row_to_slot = moe_route(ids, E)
    t_local = np.asarray(x_shards[0]).shape[0]
    w = widen(w1_shards[r], dtype)
    out = []
    for row in np.asarray(rows, dtype=np.int64):
        s = int(row_to_slot[row])
        t, k = divmod(s, topk)
        e = int(ids[t, k])
        src, lt = divmod(t, t_local)
        out.append(widen(np.asarray(x_shards[src])[lt], dtype) @ w[e])
    return np.asarray(out)


def moe_layer1_rows(h_shards, w2_shards, topk_ids, topk_weights, E: int, dtype: str,
                    o: int, rows):
    """Output_o[rows] (full H width) for sampled owner-local token rows (float64):
    for each token t, the sum over ranks r ascending and then slots k ascending
    of g[t,k] (H_r[row(t,k)] . W2_r[id[t,k]]).  Each rank's weights are widened
    once, and the products of one (r, k, expert) are taken for all sampled
    tokens at a time."""
    ids = np.asarray(topk_ids)
    g = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    T, topk = ids.shape
    R = len(h_shards)
    _, _, slot_to_row, _ = moe_route(ids, E)
    h = T // R
    toks = o * h + np.asarray(rows, dtype=np.int64)
    acc = None
    for r in range(R):
        w = widen(np.asarray(w2_shards[r]), dtype)  # [E, F/R, H]
        hs = np.asarray(h_shards[r])
        for k in range(topk):
            part = np.zeros((toks.shape[0], w.shape[2]), dtype=np.float64)
            ek = ids[toks, k]
            for e in np.unique(ek):
                sel = np.nonzero(ek == e)[0]
                hrows = widen(hs[slot_to_row[toks[sel] * topk + k]], dtype)
                part[sel] = hrows @ w[int(e)]
            v = g[toks, k][:, None] * part
            acc = v if acc is None else acc + v
    return acc


def moe_ep_layer1_rows(h, w2_ep, topk_ids, topk_weights, E: int, dtype: str, R: int, o: int, rows,
                       h_dtype: str | None = None, tp: int = 1):
    """Owner o's rows ``rows`` (full H width) of :func:`moe_ep_layer1`, token by
    token (float64): for each slot k of the token, the tp partials of its
    expert's group (t ascending), weighted by g[t,k] and added k ascending.
    ``h`` is the full grouped [T*topk x F] matrix, as there."""
    ids = np.asarray(topk_ids)
    g = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    T, topk = ids.shape
    el = E // (R // tp)
    _, _, slot_to_row, _ = moe_route(ids, E)
    hd = dtype if h_dtype is None else h_dtype
    fb = np.asarray(w2_ep[0]).shape[1]
    out = []
    for lr in np.asarray(rows, dtype=np.int64):
        tok = o * (T // R) + int(lr)
        acc = None
        for k in range(topk):
            e = int(ids[tok, k])
            grp = e // el
            hrow = widen(np.asarray(h)[slot_to_row[tok * topk + k]], hd)
            part = None
            for t in range(tp):
                v = hrow[t * fb:(t + 1) * fb] @ widen(np.asarray(w2_ep[grp * tp + t])[e % el], dtype)
                part = v if part is None else part + v
            acc = g[tok, k] * part if acc is None else acc + g[tok, k] * part
        out.append(acc)
    return np.asarray(out)
