"""The five workloads of the fused GEMM + tensor-parallel collective path.

Shapes and value distributions follow the dense TP-MLP of the FLUX paper
(Output1 = GEMM(AllGather(X), W1), Output2 = ReduceScatter(GEMM(Output1, W2)),
FLUX paper review, section "MLP 前向传播"), the Flux quick-start test shapes
(gittoolsai Flux page, section "快速开始": 4096 12288 6144 / 4096 49152 12288 /
4096 12288 49152, float16) and the COMET MoE layer (Comet article, section
"COMET 的技术原理").  R is the number of virtual tensor-parallel ranks; every
rank's shard is a separate contiguous array.

Builders return per-rank lists of numpy arrays in the storage format of
``workloads.gen`` (np.float16 for "f16", uint16 bit patterns for "bf16").
Each shard is drawn from its own stream (seed, tensor id, rank), so a shard
never depends on the others.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

from .gen import integers16, normal16, router_logits, routing, uniform16

__all__ = ["DenseAG", "DenseRS", "MoE", "CONFIGS", "ag_inputs", "rs_inputs",
           "moe_inputs", "moe_ep_inputs", "small"]


@dataclass(frozen=True)
class DenseAG:
    """AllGather + GEMM: X [M x K] row-sharded, W1 [K x N] column-sharded."""
    name: str
    R: int
    M: int
    N: int  # total columns; rank r owns N / R
    K: int
    dtype: str
    seed: int
    x_std: float = 1.0
    w_std: float = 0.02
    dist: str = "normal"  # "normal" | "uniform" | "int"

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


@dataclass(frozen=True)
class DenseRS:
    """GEMM + ReduceScatter: A [M x K] column-sharded, B [K x N] row-sharded.

    Rank r computes the partial A_r . B_r over its K / R slice; owner rank o
    receives rows [o M/R, (o+1) M/R) of the sum over r.
    """
    name: str
    R: int
    M: int
    N: int
    K: int  # total reduction length; rank r owns K / R
    dtype: str
    seed: int
    a_std: float = 1.0
    b_std: float = 0.02
    dist: str = "normal"  # "normal" | "uniform" | "int"

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


@dataclass(frozen=True)
class MoE:
    """MoE MLP with top-k routing, every expert tensor-parallel over R ranks.

    layer0: H_r = gather_by_expert(AllGather(X)) . W1_{e,r}   (F / R columns)
    layer1: Y   = ReduceScatter(sum_k g_k . (H_r . W2_{e,r}))  by token.
    """
    name: str
    R: int
    T: int
    H: int
    F: int
    E: int
    topk: int
    dtype: str
    seed: int
    zipf_s: float = 1.2
    x_std: float = 1.0
    w_std: float = 0.02
    force_empty: tuple = ()
    dist: str = "normal"

    @property
    def flops_per_layer(self) -> float:
        return 2.0 * self.T * self.topk * self.H * self.F


CONFIGS = {
    # GEMM+ReduceScatter, R=2, A [128 x 512] / B [512 x 256] split along K, U[-1, 1].
    "rs_r2_small": DenseRS("rs_r2_small", R=2, M=128, N=256, K=512, dtype="f16", seed=1,
                           dist="uniform"),
    # AllGather+GEMM dense MLP layer0, R=8.
    "ag_mlp0": DenseAG("ag_mlp0", R=8, M=4096, N=49152, K=12288, dtype="f16", seed=2),
    # GEMM+ReduceScatter dense MLP layer1, R=8.
    "rs_mlp1": DenseRS("rs_mlp1", R=8, M=4096, N=12288, K=49152, dtype="f16", seed=3),
    # decode-shaped GEMM+ReduceScatter, 70B-class down-projection, R=8, bf16.
    "rs_decode": DenseRS("rs_decode", R=8, M=128, N=8192, K=28672, dtype="bf16", seed=4),
    # MoE layer, R=8, T=4096, H=4096, F=14336, E=8, top-2, Zipf(1.2) router bias, bf16.
    "moe": MoE("moe", R=8, T=4096, H=4096, F=14336, E=8, topk=2, dtype="bf16", seed=5),
}


def _draw(key, shape, std, dtype, dist):
    if dist == "normal":
        return normal16(key, shape, std, dtype)
    if dist == "uniform":
        return uniform16(key, shape, -1.0, 1.0, dtype)
    if dist == "int":
        return integers16(key, shape, -2, 2, dtype)
    raise ValueError(dist)


def ag_inputs(c: DenseAG):
    """(x_shards R x [M/R, K], w_shards R x [K, N/R])."""
    if c.M % c.R or c.N % c.R:
        raise ValueError("M and N must divide by R")
    xs = [_draw((c.seed, 1, r), (c.M // c.R, c.K), c.x_std, c.dtype, c.dist) for r in range(c.R)]
    ws = [_draw((c.seed, 2, r), (c.K, c.N // c.R), c.w_std, c.dtype, c.dist) for r in range(c.R)]
    return xs, ws


def rs_inputs(c: DenseRS):
    """(a_shards R x [M, K/R], b_shards R x [K/R, N])."""
    if c.K % c.R or c.M % c.R:
        raise ValueError("K and M must divide by R")
    As = [_draw((c.seed, 1, r), (c.M, c.K // c.R), c.a_std, c.dtype, c.dist) for r in range(c.R)]
    Bs = [_draw((c.seed, 2, r), (c.K // c.R, c.N), c.b_std, c.dtype, c.dist) for r in range(c.R)]
    return As, Bs


def moe_inputs(c: MoE, with_h: bool = True):
    """Dict with x_shards, w1_shards, w2_shards, topk_ids, topk_weights (+ h_shards).

    x_shards  R x [T/R, H]            token rows owned by each rank
    w1_shards R x [E, H, F/R]         every expert's W1 column block of rank r
    w2_shards R x [E, F/R, H]         every expert's W2 row block of rank r
    logits    float32 [T, E]          router scores of the workload: N(0, 1) plus the
                                      Zipf(s) bias; the top-k gate (a step of the path,
                                      and of the oracle) turns them into the routing
    topk_ids  int32 [T, topk], topk_weights float32 [T, topk]
                                      a directly drawn Zipf(s) routing (no gate), the
                                      input of the layer-level tests
    h_shards  R x [T*topk, F/R]       a standalone layer1 input, N(0, 1)
    """
    if c.T % c.R or c.F % c.R:
        raise ValueError("T and F must divide by R")
    Fr = c.F // c.R
    ids, w = routing((c.seed, 9), c.T, c.E, c.topk, c.zipf_s, c.force_empty)
    d = {
        "x_shards": [_draw((c.seed, 1, r), (c.T // c.R, c.H), c.x_std, c.dtype, c.dist)
                     for r in range(c.R)],
        "w1_shards": [_draw((c.seed, 2, r), (c.E, c.H, Fr), c.w_std, c.dtype, c.dist)
                      for r in range(c.R)],
        "w2_shards": [_draw((c.seed, 3, r), (c.E, Fr, c.H), c.w_std, c.dtype, c.dist)
                      for r in range(c.R)],
        "topk_ids": ids,
        "topk_weights": w,
        "logits": router_logits((c.seed, 10), c.T, c.E, c.zipf_s, c.force_empty),
    }
    if with_h:
        d["h_shards"] = [_draw((c.seed, 4, r), (c.T * c.topk, Fr), 1.0, c.dtype, c.dist)
                         for r in range(c.R)]
    return d


def moe_ep_inputs(c: MoE, tp: int, with_h: bool = True):
    """Inputs of the MoE layer under an EP x TP split: EP = R / tp expert groups of
    tp ranks; rank r = g tp + t holds block t of group g's experts.

    x_shards  R x [T/R, H]               as in :func:`moe_inputs`
    w1_shards R x [E/EP, H, F/tp]        column block t of group g's experts' W1
    w2_shards R x [E/EP, F/tp, H]        row block t of group g's experts' W2
    topk_ids, topk_weights               as in :func:`moe_inputs`
    h_shards  R x [T*topk, F/tp]         a standalone layer1 input, N(0, 1)
    """
    if c.T % c.R or c.R % tp or c.E % (c.R // tp) or c.F % tp:
        raise ValueError("need T % R == 0, R % tp == 0, E % (R/tp) == 0, F % tp == 0")
    el, fb = c.E // (c.R // tp), c.F // tp
    ids, w = routing((c.seed, 9), c.T, c.E, c.topk, c.zipf_s, c.force_empty)
    d = {
        "x_shards": [_draw((c.seed, 1, r), (c.T // c.R, c.H), c.x_std, c.dtype, c.dist)
                     for r in range(c.R)],
        "w1_shards": [_draw((c.seed, 5, r), (el, c.H, fb), c.w_std, c.dtype, c.dist)
                      for r in range(c.R)],
        "w2_shards": [_draw((c.seed, 6, r), (el, fb, c.H), c.w_std, c.dtype, c.dist)
                      for r in range(c.R)],
        "topk_ids": ids,
        "topk_weights": w,
    }
    if with_h:
        d["h_shards"] = [_draw((c.seed, 7, r), (c.T * c.topk, fb), 1.0, c.dtype, c.dist)
                         for r in range(c.R)]
    return d


def small(c, **kw):
    """A reduced copy of a workload (same structure, smaller dims)."""
    return replace(c, **kw)
