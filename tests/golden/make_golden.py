"""Write the oracle regression fixtures in this folder.

The pages print no worked example with numbers, so these fixtures are not
the pages' values: they are written by this script, which calls only the
oracle and the seeded input generator.  They pin the oracle against
accidental change (a later edit of its arithmetic must reproduce them or
name, in its commit message, the passage that justifies the change).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import configs  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def sample_idx(seed, shape, n):
    g = np.random.default_rng(seed)
    return [g.integers(0, s, n).tolist() for s in shape]


def rs_r2_small():
    c = configs.CONFIGS["rs_r2_small"]
    As, Bs = configs.rs_inputs(c)
    out = oracle.gemm_rs(As, Bs, c.dtype)
    fx = {"source": "FLUX paper review, 'MLP 前向传播' (Output2 = ReduceScatter(GEMM(Output1, W2))); "
                    "workload: GEMM+ReduceScatter R=2, A [128x512] / B [512x256] split along K, U[-1,1], seed 1",
          "config": c.name, "ranks": []}
    for o in range(c.R):
        rows, cols = sample_idx(100 + o, out[o].shape, 64)
        fx["ranks"].append({"rows": rows, "cols": cols,
                            "values": [float(out[o][i, j]) for i, j in zip(rows, cols)],
                            "frobenius": float(np.linalg.norm(out[o]))})
    return fx


def ag_small():
    c = configs.small(configs.CONFIGS["ag_mlp0"], M=256, N=512, K=192)
    xs, ws = configs.ag_inputs(c)
    out = oracle.ag_gemm(xs, ws, c.dtype)
    fx = {"source": "FLUX paper review, 'MLP 前向传播' (Output1 = GEMM(AllGather(X), W1)); "
                    "AllGather+GEMM R=8 reduced to M=256 N=512 K=192, X N(0,1), W1 N(0,0.02), seed 2",
          "config": "ag_mlp0 reduced M=256 N=512 K=192", "ranks": []}
    for r in range(c.R):
        rows, cols = sample_idx(200 + r, out[r].shape, 32)
        fx["ranks"].append({"rows": rows, "cols": cols,
                            "values": [float(out[r][i, j]) for i, j in zip(rows, cols)],
                            "frobenius": float(np.linalg.norm(out[r]))})
    return fx


def moe_small():
    c = configs.small(configs.CONFIGS["moe"], T=64, H=64, F=128, E=8, topk=2)
    d = configs.moe_inputs(c)
    h, (counts, offsets, s2r, r2s) = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"],
                                                       c.E, c.dtype)
    y = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E, c.dtype)
    return {"source": "Comet article, 'COMET 的技术原理' (token-dimension decomposition, gather to "
                      "experts, combine by token); MoE R=8 reduced to T=64 H=64 F=128 E=8 top-2, "
                      "Zipf(1.2) expert load, bf16, seed 5",
            "config": "moe reduced T=64 H=64 F=128",
            "topk_ids": d["topk_ids"].tolist(),
            "counts": counts.tolist(), "offsets": offsets.tolist(),
            "slot_to_row": s2r.tolist(), "row_to_slot": r2s.tolist(),
            "layer0_frobenius": [float(np.linalg.norm(x)) for x in h],
            "layer1_frobenius": [float(np.linalg.norm(x)) for x in y],
            "layer1_row0_head": [float(v) for v in y[0][0, :8]]}


def gate_small():
    from workloads import gen
    L = gen.router_logits(17, 16, 8)
    ids, w = oracle.moe_topk_gate(L, 2)
    return {"source": "Comet article, 'COMET 是什么' (Mixture-of-Experts layer; the gate is the "
                      "plain top-k + softmax reading); router scores N(0,1) + Zipf(1.2) bias, "
                      "T=16 E=8 top-2, seed 17",
            "config": "gate T=16 E=8 topk=2",
            "topk_ids": ids.tolist(), "topk_weights": [[float(v) for v in row] for row in w]}


def main():
    for name, fn in [("rs_r2_small.json", rs_r2_small), ("ag_small.json", ag_small),
                     ("moe_small.json", moe_small), ("gate_small.json", gate_small)]:
        obj = fn()
        body = ",\n".join(f"{json.dumps(k)}: {json.dumps(v, ensure_ascii=False)}" for k, v in obj.items())
        with open(os.path.join(HERE, name), "w") as f:
            f.write("{\n" + body + "\n}\n")
        print("wrote", name)


if __name__ == "__main__":
    main()
