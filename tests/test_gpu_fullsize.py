"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (default options).  Every output is NaN-filled before the call and must
be finite everywhere after it (an unwritten element stays NaN); the values are
checked against the oracle on entries it computes one by one: at least one
element in every 128 x 256 output tile of every rank or owner, all four
corners of the tiles in the last tile row and column, and whole rows where the
oracle computes rows (MoE).  GPU only."""
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
TILE_M, TILE_N = 128, 256


def _ws(nbytes):
    return torch.zeros(max(nbytes, 256) // 4, dtype=torch.int32, device="cuda")


def _ok(ws):
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep


def _nan(shape, dtype):
    return torch.full(shape, float("nan"), dtype=torch_dtype(dtype), device="cuda")


def _tile_samples(seed, rows, cols, tm=TILE_M, tn=TILE_N):
    """(rows, cols) index pairs: one random element inside every tm x tn tile,
    plus the four corners of every tile of the last tile row and column."""
    g = np.random.default_rng(seed)
    mt, nt = -(-rows // tm), -(-cols // tn)
    r, c = [], []
    for i in range(mt):
        for j in range(nt):
            r0, r1 = i * tm, min(rows, (i + 1) * tm)
            c0, c1 = j * tn, min(cols, (j + 1) * tn)
            r.append(int(g.integers(r0, r1)))
            c.append(int(g.integers(c0, c1)))
            if i == mt - 1 or j == nt - 1:
                for rr in (r0, r1 - 1):
                    for cc in (c0, c1 - 1):
                        r.append(rr)
                        c.append(cc)
    return np.asarray(r), np.asarray(c)


def test_tile_samples_cover_every_tile():
    r, c = _tile_samples(0, 300, 700)
    tiles = {(a // TILE_M, b // TILE_N) for a, b in zip(r, c)}
    assert tiles == {(i, j) for i in range(3) for j in range(3)}
    assert (299, 699) in set(zip(r.tolist(), c.tolist()))
    assert r.max() < 300 and c.max() < 700


def test_ag_gemm_full_size_every_tile():
    c = configs.CONFIGS["ag_mlp0"]
    xs, w_s = configs.ag_inputs(c)
    X = [to_device(x, c.dtype) for x in xs]
    W = [to_device(w, c.dtype) for w in w_s]
    Nr = c.N // c.R
    out = [_nan((c.M, Nr), c.dtype) for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K))
    flags = torch.ones(c.R, dtype=torch.int32, device="cuda")
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, flags, ws)
    _ok(ws)
    assert torch.count_nonzero(ws).item() == 0  # the dynamic schedule leaves its area zero
    for r in range(c.R):
        assert torch.isfinite(out[r].float()).all(), f"rank {r}: unwritten (NaN) outputs"
        rows, cols = _tile_samples(100 + r, c.M, Nr)
        assert len(rows) >= (c.M // TILE_M) * (Nr // TILE_N)
        got = oracle.widen(from_device(out[r])[rows, cols], c.dtype)
        ref = oracle.ag_gemm_at(xs, w_s, c.dtype, r, rows, cols)
        check_close(got, ref, f"ag full rank {r}")


def test_gemm_rs_full_size_every_tile():
    c = configs.CONFIGS["rs_mlp1"]
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, c.dtype) for a in As]
    B = [to_device(b, c.dtype) for b in Bs]
    rows_o = c.M // c.R
    out = [_nan((rows_o, c.N), c.dtype) for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
    fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws)
    _ok(ws)
    assert torch.count_nonzero(ws).item() == 0  # counters and fp32 rows left at zero
    for o in range(c.R):
        assert torch.isfinite(out[o].float()).all(), f"owner {o}: unwritten (NaN) outputs"
        rows, cols = _tile_samples(200 + o, rows_o, c.N)
        assert len(rows) >= (rows_o // TILE_M) * (c.N // TILE_N)
        got = oracle.widen(from_device(out[o])[rows, cols], c.dtype)
        ref = oracle.gemm_rs_at(As, Bs, c.dtype, o, rows, cols)
        check_close(got, ref, f"rs full owner {o}")


def test_decode_rs_full_size_full_compare():
    c = configs.CONFIGS["rs_decode"]
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, c.dtype) for a in As]
    B = [to_device(b, c.dtype) for b in Bs]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for call in range(2):  # the second call reuses the workspace the first left at zero
        out = [_nan((c.M // c.R, c.N), c.dtype) for _ in range(c.R)]
        fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws)
        _ok(ws)
        for o in range(c.R):
            check_close(oracle.widen(from_device(out[o]), c.dtype), ref[o], f"decode call {call} owner {o}")


def _owner_rows(c, o, ids, want, seed, n=64):
    """Owner-local token rows of owner o: row 0, the last row, the tokens of
    every expert's first and last grouped slot that this owner holds, and
    random rows up to n."""
    h = c.T // c.R
    _, offsets, _, row_to_slot = want
    picks = {0, h - 1}
    for e in range(c.E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            for row in (lo, hi - 1):
                t = int(row_to_slot[row]) // c.topk
                if t // h == o:
                    picks.add(t - o * h)
    g = np.random.default_rng(seed)
    while len(picks) < n:
        picks.add(int(g.integers(0, h)))
    return np.array(sorted(picks))


def test_moe_full_size_routing_exact_and_layers_sampled():
    # the workload's routing: top-2 gate on the router scores, on the device
    # (the path) and in the oracle; ids bit-exact, then the layers
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
    H = [_nan((n, Fr), c.dtype) for _ in range(c.R)]
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
    # layer0: every grouped row written on every rank; values on the first and
    # last row of every 256-row tile of every expert, plus random rows
    off = want[1]
    picks = [np.random.default_rng(5).integers(0, n, 16)]
    for e in range(c.E):
        lo, hi = int(off[e]), int(off[e + 1])
        for t0 in range(lo, hi, 256):
            picks.append([t0, min(hi, t0 + 256) - 1])
    rows = np.unique(np.concatenate([np.asarray(p).ravel() for p in picks]))
    for r in range(c.R):
        assert torch.isfinite(H[r].float()).all(), f"layer0 rank {r}: unwritten (NaN) rows"
        got = oracle.widen(from_device(H[r])[rows], c.dtype)
        ref = oracle.moe_layer0_rows(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype, r, rows)
        check_close(got, ref, f"moe layer0 rank {r}")
    # layer1 from the standalone H input: every owner, at least 64 token rows
    # each (full width), every expert's first and last slot among them
    Y = [_nan((c.T // c.R, c.H), c.dtype) for _ in range(c.R)]
    ws1 = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_grouped_gemm_rs(c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], Hin, W2, ids, gw, offsets,
                                s2r, r2s, Y, ws1)
    _ok(ws1)
    edge_tokens = set()
    for e in range(c.E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            edge_tokens |= {int(want[3][lo]) // c.topk, int(want[3][hi - 1]) // c.topk}
    seen = set()
    for o in range(c.R):
        assert torch.isfinite(Y[o].float()).all(), f"layer1 owner {o}: unwritten (NaN) rows"
        lr = _owner_rows(c, o, ids, want, 500 + o)
        assert len(lr) >= 64
        seen |= {o * (c.T // c.R) + int(x) for x in lr}
        got = oracle.widen(from_device(Y[o])[lr], c.dtype)
        ref = oracle.moe_layer1_rows(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"],
                                     c.E, c.dtype, o, lr)
        check_close(got, ref, f"moe layer1 owner {o}")
    assert edge_tokens <= seen


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
    Y = [_nan((c.T // c.R, c.H), c.dtype) for _ in range(c.R)]
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_ep_gemm_combine(c.R, 1, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], [Hd] * c.R, W2,
                                ids, gw, None, None, None, Y, ws)
    _ok(ws)
    for o in range(c.R):
        assert torch.isfinite(Y[o].float()).all(), f"owner {o}: unwritten (NaN) rows"
    for o in (0, c.R - 1):
        lr = np.array([0, c.T // c.R - 1, 301])
        got = oracle.widen(from_device(Y[o])[lr], c.dtype)
        ref = oracle.moe_ep_layer1_rows(h, d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E,
                                        c.dtype, c.R, o, lr)
        check_close(got, ref, f"moe ep combine owner {o}")
