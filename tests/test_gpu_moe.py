"""GPU parity of the MoE path (routing, layer0 AllGather + grouped GEMM,
layer1 grouped GEMM + top-k combine + ReduceScatter) against the CPU oracle,
through the C ABI."""
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


def _ws(nbytes):
    n = max(nbytes, 256) // 4
    ws = torch.zeros(n + 64, dtype=torch.int32, device="cuda")
    off = (-ws.data_ptr()) % 256 // 4
    return ws[off:off + n]


def _i32(n):
    return torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda")


def _route_gpu(ids, E, ws=None):
    T, topk = ids.shape
    n = T * topk
    d_ids = torch.from_numpy(np.ascontiguousarray(ids)).cuda()
    counts, offsets, s2r, r2s = _i32(E), _i32(E + 1), _i32(n), _i32(n)
    fx.flux_moe_route(T, E, topk, d_ids, counts, offsets, s2r, r2s, ws)
    torch.cuda.synchronize()
    return (counts[:E].cpu().numpy(), offsets[:E + 1].cpu().numpy(), s2r[:n].cpu().numpy(),
            r2s[:n].cpu().numpy())


# ---------------------------------------------------------------- routing
@pytest.mark.parametrize("T,E,topk,empty", [(4096, 8, 2, ()), (33, 5, 3, ()), (1000, 64, 2, (3, 9)),
                                            (257, 1, 1, ()), (8192, 256, 4, ()), (0, 4, 2, ())])
def test_routing_bit_exact(T, E, topk, empty):
    ids, _ = gen.routing((77, T, E), T, E, topk, force_empty=empty) if T else \
        (np.zeros((0, topk), np.int32), None)
    got = _route_gpu(ids, E)
    want = oracle.moe_route(ids, E)
    for g, w, name in zip(got, want, ("counts", "offsets", "slot_to_row", "row_to_slot")):
        assert np.array_equal(g, w), name


def test_routing_records_invalid_expert_id():
    ids = np.array([[0, 1], [5, 2], [1, 0]], dtype=np.int32)  # 5 is outside [0, 4)
    ws = _ws(256)
    counts, offsets, s2r, r2s = _route_gpu(ids, 4, ws)
    st, _ = fx.flux_get_status(ws)
    assert st == fx.FLUX_ERR_INVALID_ARG
    assert counts.tolist() == [2, 2, 1, 0] and offsets[-1] == 5 and s2r[2] == -1


# ---------------------------------------------------------------- top-k gate
def _gate_gpu(L, topk):
    T, E = L.shape
    d_l = torch.from_numpy(np.ascontiguousarray(L, dtype=np.float32)).cuda()
    ids = torch.full((max(T * topk, 1),), -7, dtype=torch.int32, device="cuda")
    w = torch.full((max(T * topk, 1),), float("nan"), dtype=torch.float32, device="cuda")
    fx.flux_moe_topk_gate(T, E, topk, d_l, ids, w)
    torch.cuda.synchronize()
    return (ids[:T * topk].cpu().numpy().reshape(T, topk),
            w[:T * topk].cpu().numpy().astype(np.float64).reshape(T, topk))


def _check_gate(L, topk):
    ids, w = _gate_gpu(L, topk)
    rid, rw = oracle.moe_topk_gate(L, topk)
    assert np.array_equal(ids, rid)
    # expf and an fp32 sum over the k chosen scores: a few ulp relative
    assert np.allclose(w, rw, rtol=4e-6 + 2e-7 * topk, atol=1e-37)


@pytest.mark.parametrize("T,E,topk", [(4096, 8, 2), (33, 5, 3), (1000, 64, 8), (257, 1, 1),
                                      (8192, 256, 4), (64, 1024, 32), (50, 40, 40), (0, 4, 2)])
def test_gate_matches_oracle(T, E, topk):
    _check_gate(gen.router_logits((88, T, E), T, E), topk)


def test_gate_ties_and_specials():
    g = np.random.default_rng(9)
    ties = g.integers(-3, 4, size=(300, 48)).astype(np.float32)  # many equal scores
    _check_gate(ties, 6)
    sp = gen.router_logits(89, 64, 16)
    sp[0, :] = np.nan
    sp[1, 3] = np.inf
    sp[2, [1, 5]] = np.inf
    sp[3, :] = -np.inf
    sp[4, ::2] = np.nan
    sp[5, :] = 1e30
    sp[6, 7] = -1e30
    _check_gate(sp, 3)


def test_gate_feeds_the_routing():
    # gate -> route on the device equals the oracle's gate -> route
    L = gen.router_logits(90, 512, 8, force_empty=(6,))
    ids, _ = _gate_gpu(L, 2)
    got = _route_gpu(ids, 8)
    want = oracle.moe_route(oracle.moe_topk_gate(L, 2)[0], 8)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)
    assert got[0][6] == 0


# ---------------------------------------------------------------- layer0
def _layer0(c, d=None, flags=None, opts=None):
    if d is None:
        d = configs.moe_inputs(c)
    dt = c.dtype
    n = c.T * c.topk
    Fr = c.F // c.R
    X = [to_device(x, dt) for x in d["x_shards"]]
    W1 = [to_device(w, dt) for w in d["w1_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    H = [torch.full((n, Fr), float("nan"), dtype=torch_dtype(dt), device="cuda") for _ in range(c.R)]
    counts, offsets, s2r, r2s = _i32(c.E), _i32(c.E + 1), _i32(n), _i32(n)
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_ag_grouped_gemm(c.R, c.T, c.H, c.F, c.E, c.topk, DT[dt], X, W1, ids, H, counts,
                                offsets, s2r, r2s, flags, ws, opts=opts)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    routing = (counts[:c.E], offsets[:c.E + 1], s2r[:n], r2s[:n])
    return d, H, routing


@pytest.mark.parametrize("pull", [False, True], ids=["staged", "pull"])
@pytest.mark.parametrize("R,T,H,F,E,topk,dtype,empty", [
    (2, 256, 256, 640, 4, 2, "bf16", ()),      # F/R = 320: ragged n tail
    (4, 512, 192, 1024, 8, 2, "f16", (5,)),    # H = 192: ragged k tail; an empty expert
    (8, 1024, 512, 2048, 8, 2, "bf16", ()),    # the MoE workload's structure, reduced
    (1, 64, 64, 256, 3, 1, "f16", ()),
    (2, 200, 136, 256, 5, 3, "bf16", ()),      # H = 136: a 16-byte row tail in the staging copy
    (16, 1024, 256, 4096, 8, 2, "bf16", ()),   # the most ranks a call takes: 64 tokens per shard
    (4, 1000, 256, 2048, 64, 2, "f16", (3, 9, 40)),  # 64 experts, most with a partial last unit
    (4, 512, 256, 800, 8, 2, "bf16", ()),      # F/R = 200, not a multiple of 64: tiles within each rank
])
def test_layer0_matches_oracle(R, T, H, F, E, topk, dtype, empty, pull):
    # staged: every CTA first copies a share of the grouped rows, then CTA pairs
    # compute; pull: the GEMM producer gathers the rows of each tile itself
    c = configs.small(configs.CONFIGS["moe"], R=R, T=T, H=H, F=F, E=E, topk=topk, dtype=dtype,
                      seed=60 + R, force_empty=empty)
    d, Hd, routing = _layer0(c, opts={"moe_pull_gather": 1} if pull else None)
    ref, want_routing = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], E, dtype)
    for g, w in zip(routing, want_routing):
        assert np.array_equal(g.cpu().numpy(), w)
    for r in range(R):
        check_close(oracle.widen(from_device(Hd[r]), dtype), ref[r], f"layer0 rank {r}")


@pytest.mark.parametrize("case", ["layer0_ranks_side_by_side", "layer0_per_rank", "layer1"])
def test_pairs_with_an_idle_cta_match_oracle(case):
    # units whose odd CTA holds no rows, in a last n-tile of at most 128 columns
    # (none for the odd CTA): that CTA loads nothing of its own into those
    # stages.  Layer0 with F/R a multiple of 64 runs its column tiles over the
    # ranks' blocks side by side (2 x 448 = 512 + 384 columns); otherwise
    # within each rank's block (888 = 512 + 376 columns)
    if case.startswith("layer0"):
        R, Fr = (2, 448) if case == "layer0_ranks_side_by_side" else (8, 888)
        c = configs.small(configs.CONFIGS["moe"], R=R, T=2048, H=512, F=R * Fr, E=8, topk=2, seed=68)
        d, Hd, _ = _layer0(c)
        ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype)
        for r in range(c.R):
            check_close(oracle.widen(from_device(Hd[r]), c.dtype), ref[r], f"layer0 rank {r}")
    else:
        c = configs.small(configs.CONFIGS["moe"], R=8, T=2048, H=384, F=8 * 512, E=8, topk=2, seed=69)
        d = configs.moe_inputs(c)
        out, _ = _layer1(c, d)
        ref = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E,
                                c.dtype)
        for o in range(c.R):
            check_close(oracle.widen(from_device(out[o]), c.dtype), ref[o], f"layer1 owner {o}")


@pytest.mark.parametrize("stage_ctas", [1, 3, 1000])
def test_layer0_staging_split_matches_oracle(stage_ctas):
    # only the first stage_ctas CTAs copy rows; the others compute from the start
    c = configs.small(configs.CONFIGS["moe"], R=4, T=512, H=320, F=1024, E=8, topk=2, seed=67)
    d, Hd, _ = _layer0(c, opts={"moe_stage_ctas": stage_ctas})
    ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype)
    for r in range(c.R):
        check_close(oracle.widen(from_device(Hd[r]), c.dtype), ref[r], f"layer0 rank {r}")


@pytest.mark.parametrize("num_ctas", [0, 2, 6])
def test_layer0_dynamic_schedule_matches_static_bit_for_bit(num_ctas):
    # the staged layer0 claims its units from a counter (default) or takes them
    # round-robin (moe_static_schedule): a unit's arithmetic does not depend on
    # which pair runs it.  One pair (2 CTAs) and three pairs fill their
    # mailboxes with many claims each; three calls on one workspace show the
    # schedule leaves it clean for the next call
    c = configs.small(configs.CONFIGS["moe"], R=8, T=1024, H=512, F=8 * 640, E=8, topk=2, seed=65,
                      force_empty=(2,))
    d = configs.moe_inputs(c)
    base = {"num_ctas": num_ctas} if num_ctas else {}
    _, Hs, _ = _layer0(c, d=d, opts=dict(base, moe_static_schedule=1))
    ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype)
    for r in range(c.R):
        check_close(oracle.widen(from_device(Hs[r]), c.dtype), ref[r], f"static layer0 rank {r}")
    n, Fr = c.T * c.topk, c.F // c.R
    X = [to_device(x, c.dtype) for x in d["x_shards"]]
    W1 = [to_device(w, c.dtype) for w in d["w1_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    counts, offsets, s2r, r2s = _i32(c.E), _i32(c.E + 1), _i32(n), _i32(n)
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, c.R, c.T, c.H, c.F, c.E, c.topk))
    for call in range(3):
        Hd = [torch.full((n, Fr), float("nan"), dtype=torch_dtype(c.dtype), device="cuda") for _ in range(c.R)]
        fx.flux_moe_ag_grouped_gemm(c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], X, W1, ids, Hd, counts,
                                    offsets, s2r, r2s, None, ws, opts=base or None)
        st, rep = fx.flux_get_status(ws)
        assert st == fx.FLUX_OK, rep
        for r in range(c.R):
            assert torch.equal(Hd[r], Hs[r]), f"call {call} rank {r}: dynamic differs from static"


def test_layer0_accumulator_halves_match_whole_bit_for_bit():
    # the staged layer0's 256 x 512 tiles with the two-half accumulator
    # hand-over (default) and the whole one (acc_whole): same bits.  F/R = 768:
    # each rank's last column tile is 256 wide; H = 192: 3 k-slices per tile
    c = configs.small(configs.CONFIGS["moe"], R=4, T=1024, H=192, F=4 * 768, E=8, topk=2, seed=75)
    d = configs.moe_inputs(c)
    _, Ha, _ = _layer0(c, d=d)
    _, Hb, _ = _layer0(c, d=d, opts={"acc_whole": 1})
    for r in range(c.R):
        assert torch.equal(Ha[r], Hb[r]), f"rank {r}"
    ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype)
    check_close(oracle.widen(from_device(Ha[0]), c.dtype), ref[0], "layer0 halves rank 0")


def test_layer0_staged_withheld_flag_times_out_and_gpu_stays_usable():
    # token shard 1 never publishes: the staging copy of its rows gives up after
    # the timeout, the GEMM tiles waiting for those rows leave too
    c = configs.small(configs.CONFIGS["moe"], R=4, T=512, H=256, F=1024, E=8, topk=2, seed=66)
    flags = torch.tensor([1, 0, 1, 1], dtype=torch.int32, device="cuda")
    d = configs.moe_inputs(c)
    n = c.T * c.topk
    X = [to_device(x, c.dtype) for x in d["x_shards"]]
    W1 = [to_device(w, c.dtype) for w in d["w1_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    H = [torch.empty(n, c.F // c.R, dtype=torch_dtype(c.dtype), device="cuda") for _ in range(c.R)]
    counts, offsets, s2r, r2s = _i32(c.E), _i32(c.E + 1), _i32(n), _i32(n)
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_ag_grouped_gemm(c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], X, W1, ids, H, counts,
                                offsets, s2r, r2s, flags, ws, opts={"timeout_ns": 20_000_000})
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_ERR_TIMEOUT
    assert rep["where"] in ("ready flag", "staged rows"), rep
    # the same workspace (reset by flux_get_status) and GPU work normally afterwards
    flags.fill_(1)
    d2, Hd, _ = _layer0(c, d=d, flags=flags)
    ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype)
    check_close(oracle.widen(from_device(Hd[1]), c.dtype), ref[1], "after timeout")


# ---------------------------------------------------------------- layer1
def _layer1(c, d, h_dev=None, routing=None, opts=None, ws=None):
    dt = c.dtype
    n = c.T * c.topk
    Hs = h_dev if h_dev is not None else [to_device(h, dt) for h in d["h_shards"]]
    W2 = [to_device(w, dt) for w in d["w2_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    gw = torch.from_numpy(d["topk_weights"]).cuda()
    out = [torch.full((c.T // c.R, c.H), float("nan"), dtype=torch_dtype(dt), device="cuda")
           for _ in range(c.R)]
    if ws is None:
        ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    off = s2r = r2s = None
    if routing is not None:
        _, off, s2r, r2s = routing
    fx.flux_moe_grouped_gemm_rs(c.R, c.T, c.H, c.F, c.E, c.topk, DT[dt], Hs, W2, ids, gw, off, s2r,
                                r2s, out, ws, opts=opts)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    return out, ws


@pytest.mark.parametrize("R,T,H,F,E,topk,dtype,given", [
    (2, 256, 320, 512, 4, 2, "bf16", False),   # H = 320: ragged n tail
    (4, 512, 256, 768, 8, 2, "f16", True),     # F/R = 192: ragged k tail
    (8, 1024, 512, 2048, 8, 2, "bf16", True),
    (1, 96, 256, 128, 2, 2, "f16", False),
    (4, 1000, 256, 2048, 64, 2, "f16", False),  # 64 experts, most with a partial last tile
    # from 48 k-slices on: 256 x 512 tiles (H = 640: the last tile's second half
    # is past N; F/R = 3104: a 32-deep last k-slice)
    (2, 256, 640, 6208, 4, 2, "bf16", False),
    (4, 192, 1024, 12800, 8, 2, "f16", True),
    (16, 512, 256, 4096, 8, 2, "f16", True),   # the most ranks a call takes: 32 tokens per owner
])
@pytest.mark.parametrize("l1_ranks", [0, 1, 2], ids=["all-ranks-in-tmem", "per-rank-adds", "pairs-in-tmem"])
def test_layer1_matches_oracle(R, T, H, F, E, topk, dtype, given, l1_ranks):
    # l1_ranks: partials of how many ranks a CTA pair sums in TMEM before its
    # adds into the token rows (0: the default, all ranks of the expert group;
    # 1: one add per rank on 256 x 256 tiles)
    if l1_ranks > 1 and R % l1_ranks:
        pytest.skip("group size must divide the ranks")
    c = configs.small(configs.CONFIGS["moe"], R=R, T=T, H=H, F=F, E=E, topk=topk, dtype=dtype,
                      seed=80 + R)
    d = configs.moe_inputs(c)
    routing = None
    if given:
        ids = d["topk_ids"]
        routing = tuple(torch.from_numpy(a).cuda() for a in oracle.moe_route(ids, E))
    out, ws = _layer1(c, d, routing=routing, opts={"moe_l1_ranks": l1_ranks} if l1_ranks else None)
    ref = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], E, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"layer1 owner {o}")
    # the fp32 token rows, the per-tile add counts and the mailboxes (everything
    # after the routing tables) and the header, which holds the grid barrier's
    # counters, are left at zero
    a256 = lambda b: -(-b // 256) * 256  # noqa: E731
    acc_off = 256 + a256((E + 1) * 4) + a256(E * 4) + a256((E + 1) * 4) + 2 * a256(T * topk * 4)
    assert torch.count_nonzero(ws[acc_off // 4:]).item() == 0
    assert torch.count_nonzero(ws[:64]).item() == 0


def test_layer1_with_an_unrouted_slot_converts_in_the_end_pass():
    # a slot whose expert id is out of range is routed nowhere (offsets[E] <
    # T*topk), so its token's tiles never see all their adds: the layer then
    # converts the token rows in the end-of-call pass instead of at each tile's
    # last add.  The result is the layer without that slot (the oracle with
    # its gate weight 0), and the workspace is clean for the next call
    R, T, H, F, E, topk = 4, 256, 256, 1024, 4, 2
    c = configs.small(configs.CONFIGS["moe"], R=R, T=T, H=H, F=F, E=E, topk=topk, seed=95)
    d = configs.moe_inputs(c)
    n = T * topk
    ids = d["topk_ids"].copy()
    ids[5, 1] = E
    counts, off, s2r, r2s = _i32(E), _i32(E + 1), _i32(n), _i32(n)
    ws_r = _ws(256)
    fx.flux_moe_route(T, E, topk, torch.from_numpy(ids).cuda(), counts, off, s2r, r2s, ws_r)
    assert fx.flux_get_status(ws_r)[0] == fx.FLUX_ERR_INVALID_ARG
    rows = int(off[E].item())
    assert rows == n - 1
    # d["h_shards"][r][s]: rank r's layer0 row of slot s, placed in each routing's row order
    r2s_gpu = r2s[:rows].cpu().numpy()
    h_gpu = []
    for h in d["h_shards"]:
        g = np.zeros_like(h)
        g[:rows] = h[r2s_gpu]
        h_gpu.append(g)
    ids_ref = ids.copy()
    ids_ref[5, 1] = 0
    w_ref = d["topk_weights"].copy()
    w_ref[5, 1] = 0.0
    r2s_ref = oracle.moe_route(ids_ref, E)[3]
    ref = oracle.moe_layer1([h[r2s_ref] for h in d["h_shards"]], d["w2_shards"], ids_ref, w_ref, E, c.dtype)
    out, ws = _layer1(c, dict(d, topk_ids=ids), h_dev=[to_device(h, c.dtype) for h in h_gpu],
                      routing=(counts, off, s2r, r2s))
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), c.dtype), ref[o], f"unrouted slot, owner {o}")
    # the same workspace, every slot routed: the tiles are converted at their last add
    out2, _ = _layer1(c, d, ws=ws)
    ref2 = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], E, c.dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out2[o]), c.dtype), ref2[o], f"next call, owner {o}")


@pytest.mark.parametrize("l1_ranks", [0, 1, 2])
def test_layer1_integer_inputs_bit_exact(l1_ranks):
    # integer H and W2 in [-2, 2], gates 1/2: every fp32 partial, the on-chip
    # sum over ranks and the gate-weighted adds are exact, and |2 Y| <= 4 F <=
    # 1024 keeps every output exact in fp16
    c = configs.small(configs.CONFIGS["moe"], R=4, T=256, H=256, F=256, E=4, topk=2, dtype="f16",
                      dist="int", seed=93)
    d = configs.moe_inputs(c)
    d["topk_weights"] = np.full_like(d["topk_weights"], 0.5)
    out, _ = _layer1(c, d, opts={"moe_l1_ranks": l1_ranks} if l1_ranks else None)
    ref = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E,
                            c.dtype)
    for o in range(c.R):
        assert np.array_equal(oracle.widen(from_device(out[o]), c.dtype), ref[o]), o


def test_layer1_rank_group_must_divide_the_ranks():
    c = configs.small(configs.CONFIGS["moe"], R=4, T=256, H=256, F=1024, E=4, topk=2, seed=94)
    d = configs.moe_inputs(c)
    with pytest.raises(fx.FluxError, match="INVALID_ARG"):
        _layer1(c, d, opts={"moe_l1_ranks": 3})


def test_layer0_then_layer1_chained():
    c = configs.small(configs.CONFIGS["moe"], R=4, T=512, H=256, F=1024, E=8, topk=2, seed=91)
    d, Hd, routing = _layer0(c)
    out, _ = _layer1(c, d, h_dev=Hd, routing=routing)
    h_ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype)
    h_rounded = [oracle.round_to(h, c.dtype) for h in h_ref]  # layer0 stores 16-bit H
    ref = oracle.moe_layer1(h_rounded, d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E,
                            c.dtype, h_dtype="f64")
    for o in range(c.R):
        check_close(oracle.widen(from_device(out[o]), c.dtype), ref[o], f"chain owner {o}")
