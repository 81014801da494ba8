"""GPU parity of the one-call layers (dense MLP: AllGather+GEMM then
GEMM+ReduceScatter; MoE: routing, layer0, layer1) against the oracle chain,
through the C ABI.  The intermediate is stored in 16 bits by the GPU, so the
reference chain rounds it the same way before the second GEMM."""
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


def _storage(x64, dtype):
    """float64 values already rounded to `dtype`, in that 16-bit storage format."""
    if dtype == "f16":
        return x64.astype(np.float16)
    return gen.f32_to_bf16_bits(x64.astype(np.float32))


@pytest.mark.parametrize("R,M,H,F,dtype", [
    (4, 256, 512, 1024, "f16"),
    (8, 512, 256, 2048, "bf16"),
    (2, 192, 320, 640, "f16"),     # ragged tiles in both GEMMs
])
def test_mlp_one_call_matches_the_oracle_chain(R, M, H, F, dtype):
    ag = configs.small(configs.CONFIGS["ag_mlp0"], R=R, M=M, N=F, K=H, dtype=dtype, seed=70 + R)
    rs = configs.small(configs.CONFIGS["rs_mlp1"], R=R, M=M, N=H, K=F, dtype=dtype, seed=75 + R)
    xs, w1s = configs.ag_inputs(ag)
    _, w2s = configs.rs_inputs(rs)
    X = [to_device(x, dtype) for x in xs]
    W1 = [to_device(w, dtype) for w in w1s]
    W2 = [to_device(w, dtype) for w in w2s]
    h = [torch.full((M, F // R), float("nan"), dtype=torch_dtype(dtype), device="cuda")
         for _ in range(R)]
    out = [torch.full((M // R, H), float("nan"), dtype=torch_dtype(dtype), device="cuda")
           for _ in range(R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_MLP, R, M, H, F))
    fx.flux_mlp_ag_rs(R, M, H, F, DT[dtype], X, W1, h, W2, out, None, ws)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    h_ref = oracle.ag_gemm(xs, w1s, dtype)
    for r in range(R):
        check_close(oracle.widen(from_device(h[r]), dtype), h_ref[r], f"mlp h rank {r}")
    h_stored = [_storage(oracle.round_to(x, dtype), dtype) for x in h_ref]
    ref = oracle.gemm_rs(h_stored, w2s, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"mlp out owner {o}")


def test_mlp_workspace_size_is_the_gemm_rs_one():
    assert fx.flux_workspace_size(fx.FLUX_OP_MLP, 8, 512, 256, 2048) == \
        fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, 8, 512, 256, 2048)


@pytest.mark.parametrize("R,T,H,F,E,topk,dtype", [
    (4, 512, 256, 1024, 8, 2, "bf16"),
    (2, 256, 320, 640, 4, 2, "f16"),   # ragged n tails in both layers
])
def test_moe_one_call_matches_the_oracle_chain(R, T, H, F, E, topk, dtype):
    c = configs.small(configs.CONFIGS["moe"], R=R, T=T, H=H, F=F, E=E, topk=topk, dtype=dtype,
                      seed=95 + R)
    d = configs.moe_inputs(c, with_h=False)
    n, Fr = T * topk, F // R
    X = [to_device(x, dtype) for x in d["x_shards"]]
    W1 = [to_device(w, dtype) for w in d["w1_shards"]]
    W2 = [to_device(w, dtype) for w in d["w2_shards"]]
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    gw = torch.from_numpy(d["topk_weights"]).cuda()
    h = [torch.full((n, Fr), float("nan"), dtype=torch_dtype(dtype), device="cuda") for _ in range(R)]
    out = [torch.full((T // R, H), float("nan"), dtype=torch_dtype(dtype), device="cuda")
           for _ in range(R)]
    ws = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_LAYERS, R, T, H, F, E, topk))
    for _ in range(2):  # the second call reuses the workspace the first left behind
        fx.flux_moe_layers(R, T, H, F, E, topk, DT[dtype], X, W1, W2, ids, gw, h, out, None, ws)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    h_ref, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], E, dtype)
    for r in range(R):
        check_close(oracle.widen(from_device(h[r]), dtype), h_ref[r], f"moe h rank {r}")
    h_rounded = [oracle.round_to(x, dtype) for x in h_ref]
    ref = oracle.moe_layer1(h_rounded, d["w2_shards"], d["topk_ids"], d["topk_weights"], E, dtype,
                            h_dtype="f64")
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"moe out owner {o}")
