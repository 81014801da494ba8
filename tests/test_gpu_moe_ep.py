"""GPU parity of the MoE layers under an EP x TP split of the experts
(flux_moe_ep_dispatch_gemm, flux_moe_ep_gemm_combine) against the CPU oracle,
through the C ABI.  tp ranks per expert group: tp = 1 is pure expert parallel,
tp = R the tensor-parallel layout."""
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

DT = {"f16": fx.FLUX_F16, "bf16": fx.FLUX_BF16}
SENTINEL = 7.0  # rows a rank must not write keep this value


def _ws(nbytes):
    n = max(nbytes, 256) // 4
    ws = torch.zeros(n + 64, dtype=torch.int32, device="cuda")
    off = (-ws.data_ptr()) % 256 // 4
    return ws[off:off + n]


def _i32(n):
    return torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda")


def _groups(c, tp, offsets):
    """Per rank: (first row, end row) of its group's experts, column block t."""
    el = c.E // (c.R // tp)
    return [(int(offsets[(r // tp) * el]), int(offsets[(r // tp + 1) * el]), r % tp)
            for r in range(c.R)]


def _layer0(c, tp, d, shared):
    dt, n, fb = c.dtype, c.T * c.topk, c.F // tp
    X = [to_device(x, dt) for x in d["x_shards"]]
    W1 = [to_device(w, dt) for w in d["w1_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    if shared:  # ranks with the same block t share one buffer (disjoint rows)
        bufs = [torch.full((n, fb), SENTINEL, dtype=torch_dtype(dt), device="cuda")
                for _ in range(tp)]
        H = [bufs[r % tp] for r in range(c.R)]
    else:
        H = [torch.full((n, fb), SENTINEL, dtype=torch_dtype(dt), device="cuda")
             for _ in range(c.R)]
    counts, offsets, s2r, r2s = _i32(c.E), _i32(c.E + 1), _i32(n), _i32(n)
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_AG, c.R, c.T, c.H, c.F, c.E, c.topk))
    fx.flux_moe_ep_dispatch_gemm(c.R, tp, c.T, c.H, c.F, c.E, c.topk, DT[dt], X, W1, ids, H,
                                 counts, offsets, s2r, r2s, None, ws)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    routing = tuple(a[:m].cpu().numpy() for a, m in ((counts, c.E), (offsets, c.E + 1),
                                                     (s2r, n), (r2s, n)))
    return H, routing


@pytest.mark.parametrize("R,tp,T,H,F,E,topk,dtype,shared", [
    (4, 1, 512, 256, 512, 8, 2, "bf16", True),    # pure EP, one grouped buffer
    (4, 2, 256, 320, 640, 4, 2, "f16", False),    # EP 2 x TP 2, ragged n-tiles
    (4, 4, 256, 256, 1024, 8, 2, "bf16", False),  # tp = R: the tensor-parallel layout
    (8, 1, 96, 128, 256, 8, 3, "f16", False),     # one expert per rank, ragged rows
])
def test_ep_layer0_matches_oracle(R, tp, T, H, F, E, topk, dtype, shared):
    c = configs.small(configs.CONFIGS["moe"], R=R, T=T, H=H, F=F, E=E, topk=topk, dtype=dtype,
                      seed=120 + R + tp)
    d = configs.moe_ep_inputs(c, tp, with_h=False)
    Hd, routing = _layer0(c, tp, d, shared)
    ref, rref = oracle.moe_ep_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], E, dtype, tp=tp)
    for a, b, name in zip(routing, rref, ("counts", "offsets", "slot_to_row", "row_to_slot")):
        assert np.array_equal(a, b), name
    fb = F // tp
    for r, (lo, hi, t) in enumerate(_groups(c, tp, rref[1])):
        got = oracle.widen(from_device(Hd[r]), dtype)
        check_close(got[lo:hi], ref[lo:hi, t * fb:(t + 1) * fb], f"ep h rank {r}")
        if not shared:  # rows of other groups stay untouched
            assert np.all(got[:lo] == SENTINEL) and np.all(got[hi:] == SENTINEL), r


def test_ep_layer0_empty_group():
    # every token routed to experts of group 0: the other groups have no rows
    c = configs.small(configs.CONFIGS["moe"], R=4, T=128, H=128, F=256, E=8, topk=2,
                      dtype="bf16", seed=131, force_empty=(2, 3, 4, 5, 6, 7))
    d = configs.moe_ep_inputs(c, 1, with_h=False)
    Hd, routing = _layer0(c, 1, d, False)
    ref, _ = oracle.moe_ep_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, "bf16")
    got0 = oracle.widen(from_device(Hd[0]), "bf16")
    check_close(got0, ref, "ep h rank 0 (all rows)")
    for r in range(1, c.R):
        assert np.all(oracle.widen(from_device(Hd[r]), "bf16") == SENTINEL), r


def _layer1(c, tp, d, h_shards, given_routing):
    dt, n = c.dtype, c.T * c.topk
    Hs = [to_device(h, dt) for h in h_shards]
    W2 = [to_device(w, dt) for w in d["w2_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    gw = torch.from_numpy(d["topk_weights"]).cuda()
    out = [torch.full((c.T // c.R, c.H), float("nan"), dtype=torch_dtype(dt), device="cuda")
           for _ in range(c.R)]
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    if given_routing:
        _, off, s2r, r2s = oracle.moe_route(d["topk_ids"], c.E)
        rt = [torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda() for a in (off, s2r, r2s)]
    else:
        rt = [None, None, None]
    for _ in range(2):  # the second call reuses the workspace the first left behind
        fx.flux_moe_ep_gemm_combine(c.R, tp, c.T, c.H, c.F, c.E, c.topk, DT[dt], Hs, W2, ids, gw,
                                    rt[0], rt[1], rt[2], out, ws)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    return out


@pytest.mark.parametrize("R,tp,T,H,F,E,topk,dtype,given", [
    (4, 1, 512, 256, 512, 8, 2, "bf16", True),
    (4, 2, 256, 320, 640, 4, 2, "f16", False),
    (2, 2, 256, 512, 512, 4, 2, "bf16", True),
    (8, 1, 96, 136, 256, 8, 3, "f16", False),    # ragged rows and n-tiles
    # from 48 k-slices per rank on: 256 x 512 tiles
    (4, 1, 256, 384, 3072, 8, 2, "bf16", True),
    (8, 2, 128, 520, 6400, 8, 2, "f16", False),  # 8 columns in the last tile
])
def test_ep_layer1_matches_oracle(R, tp, T, H, F, E, topk, dtype, given):
    c = configs.small(configs.CONFIGS["moe"], R=R, T=T, H=H, F=F, E=E, topk=topk, dtype=dtype,
                      seed=140 + R + tp)
    d = configs.moe_ep_inputs(c, tp)
    _, offsets, _, _ = oracle.moe_route(d["topk_ids"], E)
    fb = F // tp
    h_full = np.zeros((T * topk, F), dtype=np.float64)
    for r, (lo, hi, t) in enumerate(_groups(c, tp, offsets)):
        h_full[lo:hi, t * fb:(t + 1) * fb] = oracle.widen(d["h_shards"][r], dtype)[lo:hi]
    out = _layer1(c, tp, d, d["h_shards"], given)
    ref = oracle.moe_ep_layer1(h_full, d["w2_shards"], d["topk_ids"], d["topk_weights"], E, dtype,
                               R, h_dtype="f64", tp=tp)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"ep out owner {o}")


@pytest.mark.parametrize("R,tp,T,H,F,E,topk,dtype", [
    (4, 1, 512, 256, 512, 8, 2, "bf16"),
    (4, 2, 256, 320, 640, 8, 2, "f16"),
])
def test_ep_chain_matches_oracle(R, tp, T, H, F, E, topk, dtype):
    # layer0 into shared per-block buffers, then layer1 from them with layer0's routing
    c = configs.small(configs.CONFIGS["moe"], R=R, T=T, H=H, F=F, E=E, topk=topk, dtype=dtype,
                      seed=150 + R + tp)
    d = configs.moe_ep_inputs(c, tp, with_h=False)
    Hd, routing = _layer0(c, tp, d, True)
    W2 = [to_device(w, dtype) for w in d["w2_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    gw = torch.from_numpy(d["topk_weights"]).cuda()
    rt = [torch.from_numpy(a).cuda() for a in routing[1:]]
    out = [torch.full((T // R, H), float("nan"), dtype=torch_dtype(dtype), device="cuda")
           for _ in range(R)]
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_RS, R, T, H, F, E, topk))
    fx.flux_moe_ep_gemm_combine(R, tp, T, H, F, E, topk, DT[dtype], Hd, W2, ids, gw, rt[0], rt[1],
                                rt[2], out, ws)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    h_ref, _ = oracle.moe_ep_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], E, dtype, tp=tp)
    ref = oracle.moe_ep_layer1(oracle.round_to(h_ref, dtype), d["w2_shards"], d["topk_ids"],
                               d["topk_weights"], E, dtype, R, h_dtype="f64", tp=tp)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"ep chain owner {o}")
