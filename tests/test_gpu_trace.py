"""Per-unit trace of the fused kernels (flux_opts_t.trace): every unit of the
schedule is recorded by every CTA of the region that ran it, and each
record's stamps follow the order of the pipeline (producer, MMA, epilogue).
GPU only."""
import numpy as np
import pytest

import oracle
from tests.parity import check_close
from workloads import configs
from workloads.torch_io import from_device, to_device, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reducescatter_tcgen05_tmem_gb300 as fx  # noqa: E402
from reducescatter_tcgen05_tmem_gb300 import trace as ftrace  # noqa: E402

DT = {"f16": fx.FLUX_F16, "bf16": fx.FLUX_BF16}


def _ws(nbytes):
    return torch.zeros(max(nbytes, 256) // 4, dtype=torch.int32, device="cuda")


def _check_records(t, units, per_unit, drains=None):
    """Every unit (claim) id in [0, units) recorded `per_unit` times (CTAs x the
    claim's items; an array: per id); the stamps of every record in pipeline
    order, and per CTA in item order.  `drains`: how many of all records hand
    an accumulator to the epilogue (default: every one)."""
    tag_ok = t["unit"] >= 0
    ids, counts = np.unique(t["unit"][tag_ok], return_counts=True)
    assert np.array_equal(ids, np.arange(units)), "units missing from the trace"
    assert np.all(counts == per_unit), np.unique(counts)
    n_drained = 0
    for b in range(t["grid"]):
        items = np.nonzero(tag_ok[b])[0]
        if items.size == 0:
            continue
        assert np.array_equal(items, np.arange(items.size)), f"CTA {b}: gap in its records"
        ps, pe = t["prod_start"][b, items], t["prod_end"][b, items]
        assert np.all(ps > 0) and np.all(pe >= ps), f"CTA {b}: producer stamps"
        assert np.all(np.diff(ps) >= 0), f"CTA {b}: items out of order"
        ef, ee = t["epi_full"][b, items], t["epi_end"][b, items]
        d = ef > 0  # the items that handed their accumulator to the epilogue
        n_drained += int(np.sum(d))
        if drains is None:
            assert np.all(d), f"CTA {b}: epilogue records"
        assert np.all(ee[d] >= ef[d]), f"CTA {b}: epilogue stamps"
        assert np.all(ef[d] >= ps[d]), f"CTA {b}: accumulator full before its loads began"
        ma, mf, me = t["mma_acc"][b, items], t["mma_first"][b, items], t["mma_end"][b, items]
        if np.any(me):  # the CTA that issues its pair's MMAs
            assert np.all(mf >= ma) and np.all(me >= mf), f"CTA {b}: MMA stamps"
            assert np.all(ef[d] >= me[d] - 2000), f"CTA {b}: accumulator read before its commit"
    if drains is not None:
        assert n_drained == drains, (n_drained, drains)


def test_ag_gemm_trace_covers_every_unit_in_order():
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=8, M=2048, N=16384, K=512, dtype="bf16", seed=501)
    xs, w_s = configs.ag_inputs(c)
    X = [to_device(x, c.dtype) for x in xs]
    W = [to_device(w, c.dtype) for w in w_s]
    out = [torch.full((c.M, c.N // c.R), float("nan"), dtype=torch_dtype(c.dtype), device="cuda")
           for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K))
    tr = torch.zeros(8 + 152 * 64 * 8, dtype=torch.int64, device="cuda")
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, None, ws, opts={"trace": tr})
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    ref = oracle.ag_gemm(xs, w_s, c.dtype)
    for r in (0, c.R - 1):
        check_close(oracle.widen(from_device(out[r]), c.dtype), ref[r], f"traced ag rank {r}")
    t = ftrace.records(tr)
    info = fx.flux_launch_info(fx.FLUX_OP_AG_GEMM, DT[c.dtype])
    assert t["grid"] == info["resident_ctas"]
    # regions of 8 CTAs on 512 x 1024 units: 8 ranks x 4 m-units x 2 n-units
    _check_records(t, units=c.R * (c.M // 512) * ((c.N // c.R) // 1024), per_unit=8)


def test_gemm_rs_trace_covers_every_unit_in_order():
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=8, M=1024, N=4096, K=2048, dtype="f16", seed=502)
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, c.dtype) for a in As]
    B = [to_device(b, c.dtype) for b in Bs]
    out = [torch.full((c.M // c.R, c.N), float("nan"), dtype=torch.float16, device="cuda")
           for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
    tr = torch.zeros(8 + 152 * 64 * 8, dtype=torch.int64, device="cuda")
    fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws,
                    opts={"trace": tr, "rs_tile": 1, "rs_group": 1})
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for o in (0, c.R - 1):
        check_close(oracle.widen(from_device(out[o]), c.dtype), ref[o], f"traced rs owner {o}")
    t = ftrace.records(tr)
    # regions of 4 CTAs on 512 x 512 units: 8 ranks x 2 x 8 tiles
    _check_records(t, units=c.R * (c.M // 512) * (c.N // 512), per_unit=4)
    assert set(np.unique(t["rank"][t["unit"] >= 0])) == set(range(c.R))


def test_moe_layer0_dynamic_trace_covers_every_unit_once():
    # the staged layer0's dynamic schedule: every unit of the device tile table
    # claimed once and run by both CTAs of one pair
    c = configs.small(configs.CONFIGS["moe"], R=8, T=2048, H=512, F=8 * 896, E=8, topk=2, seed=504)
    d = configs.moe_inputs(c)
    n, Fr = c.T * c.topk, c.F // c.R
    H = [torch.full((n, Fr), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(c.R)]
    i32 = lambda k: torch.empty(k, dtype=torch.int32, device="cuda")  # noqa: E731
    counts, off, s2r, r2s = i32(c.E), i32(c.E + 1), i32(n), i32(n)
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, c.R, c.T, c.H, c.F, c.E, c.topk))
    tr = torch.zeros(8 + 152 * 64 * 8, dtype=torch.int64, device="cuda")
    fx.flux_moe_ag_grouped_gemm(c.R, c.T, c.H, c.F, c.E, c.topk, fx.FLUX_BF16,
                                [to_device(x, "bf16") for x in d["x_shards"]],
                                [to_device(w, "bf16") for w in d["w1_shards"]],
                                torch.from_numpy(d["topk_ids"]).cuda(), H, counts, off, s2r, r2s, None, ws,
                                opts={"trace": tr})
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    ref, (want_counts, _, _, _) = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, "bf16")
    for r in (0, c.R - 1):
        check_close(oracle.widen(from_device(H[r]), "bf16"), ref[r], f"traced layer0 rank {r}")
    m_units = int(sum((int(k) + 255) // 256 for k in want_counts))
    t = ftrace.records(tr)
    # (F/R = 896 is a multiple of 64: the 512-column tiles run over the ranks'
    # column blocks side by side, 14 per m-unit instead of 2 x 8 with 8
    # half-wide)
    _check_records(t, units=m_units * ((c.R * Fr + 511) // 512), per_unit=2)


def test_moe_layer1_rank_group_trace_covers_every_claim():
    # layer1 with the ranks of a tile summed in TMEM: a claim is one 256 x 512
    # tile for all R ranks, recorded by both CTAs of its pair once per rank;
    # each CTA drains once per claim
    c = configs.small(configs.CONFIGS["moe"], R=4, T=1024, H=1536, F=4 * 256, E=8, topk=2, seed=506)
    d = configs.moe_inputs(c)
    n = c.T * c.topk
    Y = [torch.full((c.T // c.R, c.H), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(c.R)]
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    tr = torch.zeros(8 + 152 * 64 * 8, dtype=torch.int64, device="cuda")
    fx.flux_moe_grouped_gemm_rs(c.R, c.T, c.H, c.F, c.E, c.topk, fx.FLUX_BF16,
                                [to_device(h, "bf16") for h in d["h_shards"]],
                                [to_device(w, "bf16") for w in d["w2_shards"]],
                                torch.from_numpy(d["topk_ids"]).cuda(), torch.from_numpy(d["topk_weights"]).cuda(),
                                None, None, None, Y, ws, opts={"trace": tr})
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    ref = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E, "bf16")
    for o in (0, c.R - 1):
        check_close(oracle.widen(from_device(Y[o]), "bf16"), ref[o], f"traced layer1 owner {o}")
    counts = np.bincount(d["topk_ids"].ravel(), minlength=c.E)
    m_units = int(sum((int(k) + 255) // 256 for k in counts))
    claims = m_units * ((c.H + 511) // 512)
    _check_records(ftrace.records(tr), units=claims, per_unit=2 * c.R, drains=2 * claims)


def test_gemm_rs_rank_group_trace_covers_every_claim():
    # rank groups of 2: every claim (a tile's pair of ranks) is recorded by the
    # 4 CTAs of its region, once per rank; the last claims (one per region)
    # go out rank by rank, one record per CTA
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=8, M=1024, N=4096, K=2048, dtype="f16", seed=505)
    As, Bs = configs.rs_inputs(c)
    out = [torch.full((c.M // c.R, c.N), float("nan"), dtype=torch.float16, device="cuda")
           for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
    tr = torch.zeros(8 + 152 * 64 * 8, dtype=torch.int64, device="cuda")
    fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], [to_device(a, c.dtype) for a in As],
                    [to_device(b, c.dtype) for b in Bs], out, ws,
                    opts={"trace": tr, "rs_tile": 1, "rs_group": 2})
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for o in (0, c.R - 1):
        check_close(oracle.widen(from_device(out[o]), c.dtype), ref[o], f"traced grouped rs owner {o}")
    t = ftrace.records(tr)
    groups = c.R * (c.M // 512) * (c.N // 512) // 2
    regions = t["grid"] // 4
    split = max(groups - regions, 0)
    claims = split + (groups - split) * 2
    per = np.array([8] * split + [4] * (claims - split))
    # drains: one per claim (a group's sum, or a single rank's partial) in each of the 4 CTAs
    _check_records(t, units=claims, per_unit=per, drains=4 * claims)


def test_trace_off_leaves_the_buffer_alone():
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=2, M=256, N=1024, K=256, dtype="f16", seed=503)
    xs, w_s = configs.ag_inputs(c)
    out = [torch.empty(c.M, c.N // c.R, dtype=torch.float16, device="cuda") for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K))
    tr = torch.zeros(8 + 8 * 152, dtype=torch.int64, device="cuda")
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, fx.FLUX_F16, [to_device(x, "f16") for x in xs],
                    [to_device(w, "f16") for w in w_s], out, None, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(tr).item() == 0
