"""GPU tests of the per-problem option table: flux_tune_* pick one of their
candidates, record it for that problem only, and calls without options then
still match the oracle."""
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


def _ws(nbytes):
    n = max(nbytes, 256) // 4
    ws = torch.zeros(n + 64, dtype=torch.int32, device="cuda")
    off = (-ws.data_ptr()) % 256 // 4
    return ws[off:off + n]


@pytest.fixture(autouse=True)
def _clean_table():
    fx.flux_tune_clear()
    yield
    fx.flux_tune_clear()


def test_tune_ag_gemm_records_one_problem():
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=4, M=512, N=2048, K=512, seed=171)
    xs, w_s = configs.ag_inputs(c)
    X = [to_device(x, c.dtype) for x in xs]
    W = [to_device(w, c.dtype) for w in w_s]
    out = [torch.empty(c.M, c.N // c.R, dtype=torch_dtype(c.dtype), device="cuda") for _ in range(c.R)]
    ws = _ws(256)
    best = fx.flux_tune_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, None, ws)
    assert best["group_n"] in (2, 4, 8, 16) and fx.flux_tune_count() == 1
    for o in out:
        o.fill_(float("nan"))
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, None, ws)  # the recorded options
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    ref = oracle.ag_gemm(xs, w_s, c.dtype)
    for r in range(c.R):
        check_close(oracle.widen(from_device(out[r]), c.dtype), ref[r], f"tuned ag rank {r}")
    fx.flux_tune_clear()
    assert fx.flux_tune_count() == 0


@pytest.mark.parametrize("R,M,N,K,dtype", [
    (8, 128, 2048, 4096, "bf16"),   # stream-K (decode) form: grid candidates
    (8, 2048, 2048, 1024, "f16"),   # cluster form: raster / rank-group candidates
])
def test_tune_gemm_rs(R, M, N, K, dtype):
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=R, M=M, N=N, K=K, dtype=dtype, seed=172)
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, dtype) for a in As]
    B = [to_device(b, dtype) for b in Bs]
    out = [torch.empty(M // R, N, dtype=torch_dtype(dtype), device="cuda") for _ in range(R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, R, M, N, K))
    best = fx.flux_tune_gemm_rs(R, M, N, K, DT[dtype], A, B, out, ws)
    assert fx.flux_tune_count() == 1
    if M == 128:
        assert best["num_ctas"] >= 0 and best["group_n"] == 0
    elif best["rs_group"]:
        # a rank-group candidate: regions of 4, the library's raster
        assert best["rs_tile"] == 1 and best["rs_group"] in (1, 2, 8) and best["group_n"] == 0
    else:
        assert best["group_n"] in (4, 8, 16) and best["tiles_per_group"] in (0, 2)
    fx.flux_gemm_rs(R, M, N, K, DT[dtype], A, B, out, ws)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    ref = oracle.gemm_rs(As, Bs, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"tuned rs owner {o}")
    # the workspace is left clean after the candidates' calls
    assert torch.count_nonzero(ws[64:]).item() == 0


def test_tune_moe_layers():
    c = configs.small(configs.CONFIGS["moe"], R=4, T=512, H=256, F=1024, E=8, topk=2, seed=173)
    d = configs.moe_inputs(c)
    n, Fr = c.T * c.topk, c.F // c.R
    X = [to_device(x, c.dtype) for x in d["x_shards"]]
    W1 = [to_device(w, c.dtype) for w in d["w1_shards"]]
    W2 = [to_device(w, c.dtype) for w in d["w2_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    gw = torch.from_numpy(d["topk_weights"]).cuda()
    H = [torch.empty(n, Fr, dtype=torch_dtype(c.dtype), device="cuda") for _ in range(c.R)]
    Y = [torch.empty(c.T // c.R, c.H, dtype=torch_dtype(c.dtype), device="cuda") for _ in range(c.R)]
    i32 = lambda k: torch.empty(k, dtype=torch.int32, device="cuda")  # noqa: E731
    counts, offsets, s2r, r2s = i32(c.E), i32(c.E + 1), i32(n), i32(n)
    ws0 = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, c.R, c.T, c.H, c.F, c.E, c.topk))
    ws1 = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, c.R, c.T, c.H, c.F, c.E, c.topk))
    b0 = fx.flux_tune_moe_layer0(c.R, c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], X, W1, ids, H,
                                 counts, offsets, s2r, r2s, None, ws0)
    b1 = fx.flux_tune_moe_layer1(c.R, c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], H, W2, ids, gw,
                                 offsets, s2r, r2s, Y, ws1)
    assert fx.flux_tune_count() == 2
    assert b0["moe_pull_gather"] == 1 or b0["group_n"] in (8, 16)
    assert b1["group_n"] in (4, 8, 16)
    # the tensor-parallel calls use the tp = R entries
    fx.flux_moe_ag_grouped_gemm(c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], X, W1, ids, H, counts,
                                offsets, s2r, r2s, None, ws0)
    fx.flux_moe_grouped_gemm_rs(c.R, c.T, c.H, c.F, c.E, c.topk, DT[c.dtype], H, W2, ids, gw, offsets,
                                s2r, r2s, Y, ws1)
    for w in (ws0, ws1):
        st, rep = fx.flux_get_status(w)
        assert st == fx.FLUX_OK, rep
    h_ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, c.dtype)
    for r in range(c.R):
        check_close(oracle.widen(from_device(H[r]), c.dtype), h_ref[r], f"tuned layer0 rank {r}")
    ref = oracle.moe_layer1([oracle.round_to(h, c.dtype) for h in h_ref], d["w2_shards"],
                            d["topk_ids"], d["topk_weights"], c.E, c.dtype, h_dtype="f64")
    for o in range(c.R):
        check_close(oracle.widen(from_device(Y[o]), c.dtype), ref[o], f"tuned layer1 owner {o}")


def test_tune_rejects_bad_arguments():
    ws = _ws(256)
    with pytest.raises(fx.FluxError):
        fx.flux_tune_ag_gemm(3, 64, 64, 64, fx.FLUX_F16, [0] * 3, [0] * 3, [0] * 3, None, ws)
    assert fx.flux_tune_count() == 0
