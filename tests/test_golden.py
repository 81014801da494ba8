"""The oracle still reproduces its committed regression fixtures (CPU only)."""
import json
import os

import numpy as np

import oracle
from workloads import configs

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_rs_r2_small_fixture():
    fx = _load("rs_r2_small.json")
    c = configs.CONFIGS["rs_r2_small"]
    out = oracle.gemm_rs(*configs.rs_inputs(c), c.dtype)
    for o, rk in enumerate(fx["ranks"]):
        got = out[o][rk["rows"], rk["cols"]]
        assert np.allclose(got, rk["values"], rtol=1e-12, atol=1e-12)
        assert np.isclose(np.linalg.norm(out[o]), rk["frobenius"], rtol=1e-12)


def test_ag_small_fixture():
    fx = _load("ag_small.json")
    c = configs.small(configs.CONFIGS["ag_mlp0"], M=256, N=512, K=192)
    out = oracle.ag_gemm(*configs.ag_inputs(c), c.dtype)
    for r, rk in enumerate(fx["ranks"]):
        assert np.allclose(out[r][rk["rows"], rk["cols"]], rk["values"], rtol=1e-12, atol=1e-12)
        assert np.isclose(np.linalg.norm(out[r]), rk["frobenius"], rtol=1e-12)


def test_moe_small_fixture():
    fx = _load("moe_small.json")
    c = configs.small(configs.CONFIGS["moe"], T=64, H=64, F=128, E=8, topk=2)
    d = configs.moe_inputs(c)
    assert d["topk_ids"].tolist() == fx["topk_ids"]
    h, (counts, offsets, s2r, r2s) = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"],
                                                       c.E, c.dtype)
    assert counts.tolist() == fx["counts"] and offsets.tolist() == fx["offsets"]
    assert s2r.tolist() == fx["slot_to_row"] and r2s.tolist() == fx["row_to_slot"]
    assert np.allclose([np.linalg.norm(x) for x in h], fx["layer0_frobenius"], rtol=1e-12)
    y = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E, c.dtype)
    assert np.allclose([np.linalg.norm(x) for x in y], fx["layer1_frobenius"], rtol=1e-12)
    assert np.allclose(y[0][0, :8], fx["layer1_row0_head"], rtol=1e-12)


def test_gate_small_fixture():
    from workloads import gen
    fx = _load("gate_small.json")
    ids, w = oracle.moe_topk_gate(gen.router_logits(17, 16, 8), 2)
    assert ids.tolist() == fx["topk_ids"]
    assert np.allclose(w, fx["topk_weights"], rtol=1e-14, atol=0)
