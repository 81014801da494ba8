"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (default options), on outputs the oracle computes one by one (or in
full where that takes seconds).  GPU only."""
import numpy as np
import pytest

import oracle
from tests.parity import check_close
from workloads import configs, gen
from workloads.torch_io import from_device, to_device, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reducescatter_tcgen05_tmem_gb300 as fx  # noqa: E402

DT = {"f16": fx.FLUX_F16, "bf16": fx.FLUX_BF16}
SAMPLES = 48


def _ws(nbytes):
    return torch.zeros(max(nbytes, 256) // 4, dtype=torch.int32, device="cuda")


def _ok(ws):
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep


def _pairs(seed, rows, cols, n=SAMPLES):
    g = np.random.default_rng(seed)
    # include the corners of the tile grid, then random positions
    r = np.concatenate([[0, rows - 1, rows // 2], g.integers(0, rows, n - 3)])
    c = np.concatenate([[0, cols - 1, cols // 3], g.integers(0, cols, n - 3)])
    return r, c


def test_ag_gemm_full_size_sampled():
    c = configs.CONFIGS["ag_mlp0"]
    xs, w_s = configs.ag_inputs(c)
    X = [to_device(x, c.dtype) for x in xs]
    W = [to_device(w, c.dtype) for w in w_s]
    out = [torch.empty(c.M, c.N // c.R, dtype=torch.float16, device="cuda") for _ in range(c.R)]
    ws = _ws(256)
    flags = torch.ones(c.R, dtype=torch.int32, device="cuda")
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, flags, ws)
    _ok(ws)
    for r in range(c.R):
        rows, cols = _pairs(100 + r, c.M, c.N // c.R)
        got = oracle.widen(from_device(out[r])[rows, cols], c.dtype)
        ref = oracle.ag_gemm_at(xs, w_s, c.dtype, r, rows, cols)
        check_close(got, ref, f"ag full rank {r}")
        assert torch.isfinite(out[r].float()).all()


def test_gemm_rs_full_size_sampled():
    c = configs.CONFIGS["rs_mlp1"]
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, c.dtype) for a in As]
    B = [to_device(b, c.dtype) for b in Bs]
    out = [torch.empty(c.M // c.R, c.N, dtype=torch.float16, device="cuda") for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
    fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws)
    _ok(ws)
    for o in range(c.R):
        rows, cols = _pairs(200 + o, c.M // c.R, c.N, 24)
        got = oracle.widen(from_device(out[o])[rows, cols], c.dtype)
        ref = oracle.gemm_rs_at(As, Bs, c.dtype, o, rows, cols)
        check_close(got, ref, f"rs full owner {o}")
        assert torch.isfinite(out[o].float()).all()
    assert torch.count_nonzero(ws).item() == 0


def test_decode_rs_full_size_full_compare():
    c = configs.CONFIGS["rs_decode"]
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, c.dtype) for a in As]
    B = [to_device(b, c.dtype) for b in Bs]
    out = [torch.empty(c.M // c.R, c.N, dtype=torch.bfloat16, device="cuda") for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
    for _ in range(2):  # the second call reuses the workspace the first left at zero
        fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws)
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for o in range(c.R):
        check_close(oracle.widen(from_device(out[o]), c.dtype), ref[o], f"decode owner {o}")


def test_moe_full_size_routing_exact_and_layers_sampled():
    # the workload's routing: top-2 gate on the router scores, on the device
    # (the path) and in the oracle; ids bit-exact, the layers then sampled
    c = configs.CONFIGS["moe"]
    d = configs.moe_inputs(c)
    n, Fr = c.T * c.topk, c.F // c.R
    X = [to_device(x, c.dtype) for x in d["x_shards"]]
    W1 = [to_device(w, c.dtype) for w in d["w1_shards"]]
    W2 = [to_device(w, c.dtype) for w in d["w2_shards"]]
    Hin = [to_device(h, c.dtype) for h in d["h_shards"]]
    ids = torch.empty(c.T, c.topk, dtype=torch.int32, device="cuda")
    gw = torch.empty(c.T, c.topk, dtype=torch.float32, device="cuda")
    fx.flux_moe_topk_gate(c.T, c.E, c.topk, torch.from_numpy(d["logits"]).cuda(), ids, gw)
    ref_ids, ref_gw = oracle.moe_topk_gate(d["logits"], c.topk)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.allclose(gw.cpu().numpy(), ref_gw, rtol=5e-6, atol=1e-37)
    d["topk_ids"], d["topk_weights"] = ref_ids, ref_gw  # the oracle continues from its own gate
    H = [torch.empty(n, Fr, dtype=torch.bfloat16, device="cuda") for _ in range(c.R)]
    counts = torch.empty(c.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(c.E + 1, dtype=torch.int32, device="cuda")
    s2r = torch.empty(n, dtype=torch.int32, device="cuda")
    r2s = torch.empty(n, dtype=torch.int32, device="cuda")
    ws0 = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, c.R, c.T, c.H, c.F, c.E, c.topk))
    flags = torch.ones(c.R, dtype=torch.int32, device="cuda")
    fx.flux_moe_ag_grouped_gemm(c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], X, W1, ids, H, counts,
                                offsets, s2r, r2s, flags, ws0)
    _ok(ws0)
    want = oracle.moe_route(d["topk_ids"], c.E)
    for g, w in zip((counts, offsets, s2r, r2s), want):
        assert np.array_equal(g.cpu().numpy(), w)
    # layer0 on sampled grouped rows (every expert's first and last row included)
    off = want[1]
    rows = np.unique(np.concatenate([off[:-1], np.maximum(off[1:] - 1, 0),
                                     np.random.default_rng(5).integers(0, n, 24)]))
    rows = rows[rows < n]
    for r in (0, c.R - 1):
        got = oracle.widen(from_device(H[r])[rows], c.dtype)
        ref = oracle.moe_layer0_rows(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype, r, rows)
        check_close(got, ref, f"moe layer0 rank {r}")
    # layer1 from the standalone H input, sampled owner rows (full width)
    Y = [torch.empty(c.T // c.R, c.H, dtype=torch.bfloat16, device="cuda") for _ in range(c.R)]
    ws1 = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_grouped_gemm_rs(c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], Hin, W2, ids, gw, offsets,
                                s2r, r2s, Y, ws1)
    _ok(ws1)
    for o in (0, 3, c.R - 1):
        lr = np.array([0, 1, c.T // c.R - 1, 77])
        got = oracle.widen(from_device(Y[o])[lr], c.dtype)
        ref = oracle.moe_layer1_rows(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"],
                                     c.E, c.dtype, o, lr)
        check_close(got, ref, f"moe layer1 owner {o}")


def test_moe_ep_combine_full_size_sampled():
    # expert parallel, one expert per rank (tp = 1): each rank reduces over the
    # whole F = 14336 (224 k-slices, the 256 x 512 tile form); every rank reads
    # the same grouped H [T*topk x F]
    c = configs.CONFIGS["moe"]
    d = configs.moe_ep_inputs(c, 1, with_h=False)
    del d["w1_shards"]
    n = c.T * c.topk
    h = gen.normal16((c.seed, 23), (n, c.F), 1.0, c.dtype)
    Hd = to_device(h, c.dtype)
    W2 = [to_device(w, c.dtype) for w in d["w2_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    gw = torch.from_numpy(d["topk_weights"]).cuda()
    Y = [torch.full((c.T // c.R, c.H), float("nan"), dtype=torch_dtype(c.dtype), device="cuda")
         for _ in range(c.R)]
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_ep_gemm_combine(c.R, 1, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], [Hd] * c.R, W2,
                                ids, gw, None, None, None, Y, ws)
    _ok(ws)
    for o in (0, c.R - 1):
        lr = np.array([0, c.T // c.R - 1, 301])
        got = oracle.widen(from_device(Y[o])[lr], c.dtype)
        ref = oracle.moe_ep_layer1_rows(h, d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E,
                                        c.dtype, c.R, o, lr)
        check_close(got, ref, f"moe ep combine owner {o}")
