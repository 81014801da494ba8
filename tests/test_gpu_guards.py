"""Every write of a call stays inside its outputs.

All outputs of a call are cut out of one flat buffer, with guard bands that
hold a sentinel before, between and after them; each guard is at least 256
full rows of the output after it, so a tile that runs past a ragged row tail
or an owner chunk smaller than a tile lands in a guard.  After the call the
guards must still hold the sentinel bit for bit, and the outputs must match
the oracle.  This stands in for a device memory checker on the epilogues'
tail handling: plain GEMM, AllGather + GEMM, the three forms of GEMM +
ReduceScatter (4-CTA cluster reduction, stream-K, whole units on the dynamic
schedule) and both MoE layers.
"""
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
SENTINEL = 7.0  # exact in fp16 and bf16
ALIGN = 128     # elements: 256 bytes of 16-bit values


def _ws(nbytes):
    n = max(nbytes, 256) // 4
    ws = torch.zeros(n + 64, dtype=torch.int32, device="cuda")
    off = (-ws.data_ptr()) % 256 // 4
    return ws[off:off + n]


class Guarded:
    """Outputs of the given (rows, cols) shapes inside one sentinel-filled buffer."""

    def __init__(self, shapes, dtype):
        up = lambda n: -(-n // ALIGN) * ALIGN  # noqa: E731
        spans, off = [], 0
        for rows, cols in shapes:
            off += up(max(256 * cols, 2048))          # guard before this output
            spans.append((off, rows, cols))
            off += up(rows * cols)
        total = off + up(max(256 * shapes[-1][1], 2048))  # guard after the last one
        self.flat = torch.full((total + ALIGN,), SENTINEL, dtype=torch_dtype(dtype), device="cuda")
        base = (-self.flat.data_ptr()) % 256 // 2
        self.flat = self.flat[base:base + total]
        self.spans = spans
        self.outs = [self.flat[o:o + r * c].view(r, c) for o, r, c in spans]

    def check_guards(self, what):
        inside = np.zeros(self.flat.numel(), dtype=bool)
        for o, r, c in self.spans:
            inside[o:o + r * c] = True
        host = self.flat.float().cpu().numpy()
        bad = np.flatnonzero(~inside & (host != SENTINEL))
        assert bad.size == 0, f"{what}: {bad.size} guard elements written, first at {bad[:4]}"


def _ok(ws):
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep


@pytest.mark.parametrize("M,N,K,dtype", [(300, 264, 200, "f16"), (129, 1000, 64, "bf16")])
def test_gemm_writes_stay_inside(M, N, K, dtype):
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=1, M=M, N=N, K=K, dtype=dtype, seed=301)
    xs, w_s = configs.ag_inputs(c)
    g = Guarded([(M, N)], dtype)
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM, 1, M, N, K))
    fx.flux_gemm(M, N, K, DT[dtype], to_device(xs[0], dtype), to_device(w_s[0], dtype), g.outs[0], ws)
    _ok(ws)
    g.check_guards("gemm")
    ref = oracle.gemm(oracle.widen(xs[0], dtype), oracle.widen(w_s[0], dtype))
    check_close(oracle.widen(from_device(g.outs[0]), dtype), ref, "gemm")


@pytest.mark.parametrize("R,M,N,K,dtype", [
    (8, 320, 576, 200, "f16"),      # 40-row shards, 72 columns per rank
    (8, 1088, 2112, 136, "bf16"),   # 136-row shards, 264 columns per rank: ragged 512-wide units
])
def test_ag_gemm_writes_stay_inside(R, M, N, K, dtype):
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=R, M=M, N=N, K=K, dtype=dtype, seed=302)
    xs, w_s = configs.ag_inputs(c)
    g = Guarded([(M, N // R)] * R, dtype)
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, R, M, N, K))
    fx.flux_ag_gemm(R, M, N, K, DT[dtype], [to_device(x, dtype) for x in xs],
                    [to_device(w, dtype) for w in w_s], g.outs, None, ws)
    _ok(ws)
    g.check_guards("ag_gemm")
    ref = oracle.ag_gemm(xs, w_s, dtype)
    for r in range(R):
        check_close(oracle.widen(from_device(g.outs[r]), dtype), ref[r], f"ag rank {r}")


@pytest.mark.parametrize("R,M,N,K,dtype,rs_tile", [
    (4, 96, 264, 512, "f16", 0),     # at most 128 rows, 4 ranks: 4-CTA cluster reduction, 24-row owners
    (2, 64, 1000, 4096, "bf16", 0),  # few tiles: stream-K, 32-row owners, ragged last n-tile
    (8, 1088, 2056, 256, "f16", 1),  # 648 rank tiles: whole units, regions of 4, 136-row owners
    (8, 1088, 2056, 256, "f16", 2),  # the same on regions of 8 (256 x 256 pair tiles)
    (8, 1088, 2056, 256, "f16", 3),  # regions of 4, tile-major (a tile's ranks back to back)
])
def test_gemm_rs_writes_stay_inside(R, M, N, K, dtype, rs_tile):
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=R, M=M, N=N, K=K, dtype=dtype, seed=303)
    As, Bs = configs.rs_inputs(c)
    g = Guarded([(M // R, N)] * R, dtype)
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, R, M, N, K))
    fx.flux_gemm_rs(R, M, N, K, DT[dtype], [to_device(a, dtype) for a in As],
                    [to_device(b, dtype) for b in Bs], g.outs, ws,
                    opts={"rs_tile": rs_tile} if rs_tile else None)
    _ok(ws)
    g.check_guards("gemm_rs")
    ref = oracle.gemm_rs(As, Bs, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(g.outs[o]), dtype), ref[o], f"rs owner {o}")


def _i32(n):
    return torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("R,T,H,F,E,dtype", [
    (4, 512, 192, 1024, 8, "f16"),   # F/R = 256: half of a 512-wide tile past the columns
    (2, 200, 136, 640, 5, "bf16"),   # F/R = 320, ragged experts
])
def test_moe_layers_write_stay_inside(R, T, H, F, E, dtype):
    topk = 2
    c = configs.small(configs.CONFIGS["moe"], R=R, T=T, H=H, F=F, E=E, topk=topk, dtype=dtype,
                      seed=304)
    d = configs.moe_inputs(c)
    n, Fr = T * topk, F // R
    ids = torch.from_numpy(d["topk_ids"]).cuda()
    gw = torch.from_numpy(d["topk_weights"]).cuda()
    # layer0: grouped rows [T*topk x F/R] per rank
    g0 = Guarded([(n, Fr)] * R, dtype)
    counts, offsets, s2r, r2s = _i32(E), _i32(E + 1), _i32(n), _i32(n)
    ws0 = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, R, T, H, F, E, topk))
    fx.flux_moe_ag_grouped_gemm(R, T, H, F, E, topk, DT[dtype], [to_device(x, dtype) for x in d["x_shards"]],
                                [to_device(w, dtype) for w in d["w1_shards"]], ids, g0.outs, counts,
                                offsets, s2r, r2s, None, ws0)
    _ok(ws0)
    g0.check_guards("moe layer0")
    ref0, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], E, dtype)
    for r in range(R):
        check_close(oracle.widen(from_device(g0.outs[r]), dtype), ref0[r], f"layer0 rank {r}")
    # layer1: owner rows [T/R x H], fed by the generator's H
    g1 = Guarded([(T // R, H)] * R, dtype)
    ws1 = _ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, R, T, H, F, E, topk))
    fx.flux_moe_grouped_gemm_rs(R, T, H, F, E, topk, DT[dtype], [to_device(h, dtype) for h in d["h_shards"]],
                                [to_device(w, dtype) for w in d["w2_shards"]], ids, gw, None, None,
                                None, g1.outs, ws1)
    _ok(ws1)
    g1.check_guards("moe layer1")
    ref1 = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], E, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(g1.outs[o]), dtype), ref1[o], f"layer1 owner {o}")
