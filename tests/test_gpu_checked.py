"""The checked build of the library (libflux_gb300_checked.so, -DFLUX_CHECKS=1):
every TMA coordinate and global store or add of the kernels is checked.  In a
child process that loads it (FLUX_CHECKED=1), each op runs on inputs that
reach its ragged tails, its cluster and stream-K forms and its MoE boundaries;
no check may fire and the results must match the oracle.  The deliberate
probe must be reported as a failed check, and the GPU must stay usable.
GPU only."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import json, sys
import numpy as np
import torch
import oracle
import reducescatter_tcgen05_tmem_gb300 as fx
from tests.parity import check_close
from workloads import configs, gen
from workloads.torch_io import from_device, to_device, torch_dtype

assert fx.CHECKED and fx.flux_checks_enabled(), "the checked library is not the one loaded"
DT = {"f16": fx.FLUX_F16, "bf16": fx.FLUX_BF16}
done = []

def ws_of(n):
    return torch.zeros(max(n, 256) // 4, dtype=torch.int32, device="cuda")

def ok(ws, what):
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, (what, rep)
    done.append(what)

# AllGather + GEMM (pull and push), ragged shards and tails
for push in (0, 1):
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=8, M=320, N=576, K=200, seed=701)
    xs, w_s = configs.ag_inputs(c)
    out = [torch.full((c.M, c.N // c.R), float("nan"), dtype=torch.float16, device="cuda") for _ in range(c.R)]
    op = fx.FLUX_OP_AG_GEMM_PUSH if push else fx.FLUX_OP_AG_GEMM
    ws = ws_of(fx.flux_workspace_size(op, c.R, c.M, c.N, c.K))
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, fx.FLUX_F16, [to_device(x, "f16") for x in xs],
                    [to_device(w, "f16") for w in w_s], out, None, ws, opts={"ag_push": push} if push else None)
    ok(ws, f"ag push={push}")
    ref = oracle.ag_gemm(xs, w_s, "f16")
    for r in range(c.R):
        check_close(oracle.widen(from_device(out[r]), "f16"), ref[r], f"checked ag rank {r}")

# GEMM + ReduceScatter: whole units (three forms; rank groups summed in TMEM, and groups of
# all ranks stored as 16-bit), stream-K, cluster form; plain GEMM split-K
for (R, M, N, K, dt, o) in [(8, 1088, 2056, 256, "f16", {}), (8, 1088, 2056, 256, "f16", {"rs_tile": 2}),
                            (8, 1088, 2056, 256, "f16", {"rs_tile": 3}), (2, 64, 1000, 4096, "bf16", {}),
                            (8, 128, 2048, 4096, "bf16", {}), (4, 256, 512, 1024, "f16", {"deterministic_rs": 1}),
                            (8, 1024, 2056, 4096, "bf16", {"rs_group": 8})]:
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=R, M=M, N=N, K=K, dtype=dt, seed=702)
    As, Bs = configs.rs_inputs(c)
    out = [torch.full((M // R, N), float("nan"), dtype=torch_dtype(dt), device="cuda") for _ in range(R)]
    ws = ws_of(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, R, M, N, K))
    fx.flux_gemm_rs(R, M, N, K, DT[dt], [to_device(a, dt) for a in As], [to_device(b, dt) for b in Bs], out,
                    ws, opts=o or None)
    ok(ws, f"rs {R}x{M}x{N}x{K} {o}")
    ref = oracle.gemm_rs(As, Bs, dt)
    for r in range(R):
        check_close(oracle.widen(from_device(out[r]), dt), ref[r], f"checked rs owner {r}")
A = gen.normal16((703, 1), (128, 4096), 1.0, "bf16")
B = gen.normal16((703, 2), (4096, 2048), 0.02, "bf16")
C = torch.full((128, 2048), float("nan"), dtype=torch.bfloat16, device="cuda")
ws = ws_of(fx.flux_workspace_size(fx.FLUX_OP_GEMM, 1, 128, 2048, 4096))
fx.flux_gemm(128, 2048, 4096, fx.FLUX_BF16, to_device(A, "bf16"), to_device(B, "bf16"), C, ws)
ok(ws, "plain gemm split-K")
check_close(oracle.widen(from_device(C), "bf16"), oracle.gemm(oracle.widen(A, "bf16"), oracle.widen(B, "bf16")),
            "checked plain gemm")

# MoE layers (staged layer0 with column tiles over the ranks' blocks side by side and within
# each rank's block, pull layer0; layer1 per rank and with ranks summed on chip), empty expert
for pull, l1, Fr in ((0, 0, 448), (1, 4, 448), (0, 1, 440)):
    c = configs.small(configs.CONFIGS["moe"], R=4, T=512, H=320, F=4 * Fr, E=8, topk=2, seed=704,
                      force_empty=(5,))
    d = configs.moe_inputs(c)
    n, Fr = c.T * c.topk, c.F // c.R
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    gw = torch.from_numpy(d["topk_weights"]).cuda()
    H = [torch.full((n, Fr), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(c.R)]
    cnt = torch.empty(c.E, dtype=torch.int32, device="cuda")
    off = torch.empty(c.E + 1, dtype=torch.int32, device="cuda")
    s2r = torch.empty(n, dtype=torch.int32, device="cuda")
    r2s = torch.empty(n, dtype=torch.int32, device="cuda")
    ws0 = ws_of(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_ag_grouped_gemm(c.R, c.T, c.H, c.F, c.E, c.topk, fx.FLUX_BF16,
                                [to_device(x, "bf16") for x in d["x_shards"]],
                                [to_device(w, "bf16") for w in d["w1_shards"]], ids, H, cnt, off, s2r, r2s,
                                None, ws0, opts={"moe_pull_gather": pull} if pull else None)
    ok(ws0, f"moe layer0 pull={pull}")
    h_ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, "bf16")
    for r in range(c.R):
        check_close(oracle.widen(from_device(H[r]), "bf16"), h_ref[r], f"checked layer0 rank {r}")
    Y = [torch.full((c.T // c.R, c.H), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(c.R)]
    ws1 = ws_of(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_grouped_gemm_rs(c.R, c.T, c.H, c.F, c.E, c.topk, fx.FLUX_BF16,
                                [to_device(h, "bf16") for h in d["h_shards"]],
                                [to_device(w, "bf16") for w in d["w2_shards"]], ids, gw, off, s2r, r2s, Y, ws1,
                                opts={"moe_l1_ranks": l1} if l1 else None)
    ok(ws1, f"moe layer1 ranks-on-chip={l1}")
    y_ref = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E, "bf16")
    for r in range(c.R):
        check_close(oracle.widen(from_device(Y[r]), "bf16"), y_ref[r], f"checked layer1 owner {r}")

# the probe: one deliberate failed check, reported; the next call is clean
c = configs.small(configs.CONFIGS["rs_mlp1"], R=4, M=512, N=512, K=512, seed=705)
As, Bs = configs.rs_inputs(c)
A_ = [to_device(a, "f16") for a in As]
B_ = [to_device(b, "f16") for b in Bs]
out = [torch.empty(c.M // c.R, c.N, dtype=torch.float16, device="cuda") for _ in range(c.R)]
ws = ws_of(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
fx.flux_gemm_rs(c.R, c.M, c.N, c.K, fx.FLUX_F16, A_, B_, out, ws, opts={"debug_probe": 1234, "timeout_ns": 20_000_000})
st, rep = fx.flux_get_status(ws)
probe = {"status": st, "report": rep}
fx.flux_gemm_rs(c.R, c.M, c.N, c.K, fx.FLUX_F16, A_, B_, out, ws)
ok(ws, "after the probe")
ref = oracle.gemm_rs(As, Bs, "f16")
for r in range(c.R):
    check_close(oracle.widen(from_device(out[r]), "f16"), ref[r], f"after probe owner {r}")
print("RESULT " + json.dumps({"done": done, "probe": probe}))
'''


def test_checked_build_runs_every_op_clean_and_reports_the_probe():
    import reducescatter_tcgen05_tmem_gb300 as fx
    assert not fx.flux_checks_enabled()  # this process has the regular build
    env = dict(os.environ, FLUX_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    assert len(res["done"]) == 17, res["done"]  # 2 AG, 7 GEMM-RS, 1 plain GEMM, 6 MoE, 1 after the probe
    assert res["probe"]["status"] == fx.FLUX_ERR_INVALID_ARG
    rep = res["probe"]["report"]
    assert rep["where"] == "check" and rep["arg0"] == 15 and rep["arg1"] == 1234, rep
