"""GPU parity of the dense ops (plain GEMM, AllGather+GEMM, GEMM+ReduceScatter)
against the float64 CPU oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from tests.parity import check_close
from workloads import configs, gen
from workloads.torch_io import from_device, to_device, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines skip the module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reducescatter_tcgen05_tmem_gb300 as fx  # noqa: E402

DT = {"f16": fx.FLUX_F16, "bf16": fx.FLUX_BF16}


def _ws(nbytes):
    ws = torch.zeros(max(nbytes, 256) // 4 + 64, dtype=torch.int32, device="cuda")
    # 256-byte aligned view
    off = (-ws.data_ptr()) % 256 // 4
    return ws[off:off + max(nbytes, 256) // 4]


def _out(rows, cols, dtype):
    return torch.full((rows, cols), float("nan"), dtype=torch_dtype(dtype), device="cuda")


def _ok(ws):
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep


# ---------------------------------------------------------------- plain GEMM
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 264, 200), (1, 8, 8), (257, 520, 1032),
                                   (512, 768, 4096)])
def test_gemm_matches_oracle(dtype, M, N, K):
    A = gen.normal16((7, 1), (M, K), 1.0, dtype)
    B = gen.normal16((7, 2), (K, N), 0.05, dtype)
    C = _out(M, N, dtype)
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM, 1, M, N, K))
    fx.flux_gemm(M, N, K, DT[dtype], to_device(A, dtype), to_device(B, dtype), C, ws)
    _ok(ws)
    ref = oracle.gemm(oracle.widen(A, dtype), oracle.widen(B, dtype))
    check_close(oracle.widen(from_device(C), dtype), ref, f"gemm {M}x{N}x{K} {dtype}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gemm_integer_inputs_are_bit_exact(dtype):
    # |partial sums| <= 2*2*64 = 256: exact in fp32 and in both 16-bit formats
    M, N, K = 200, 320, 64
    A = gen.integers16((8, 1), (M, K), -2, 2, dtype)
    B = gen.integers16((8, 2), (K, N), -2, 2, dtype)
    C = _out(M, N, dtype)
    ws = _ws(256)
    fx.flux_gemm(M, N, K, DT[dtype], to_device(A, dtype), to_device(B, dtype), C, ws)
    _ok(ws)
    ref = oracle.gemm(oracle.widen(A, dtype), oracle.widen(B, dtype))
    assert np.array_equal(oracle.widen(from_device(C), dtype), ref)


@pytest.mark.parametrize("M,N,K,dtype", [
    (128, 8192, 8192, "bf16"),   # 8 K slices, 32 n-tiles on 4-CTA clusters
    (64, 2048, 4096, "f16"),     # 8 slices, 8-row chunks
    (100, 1000, 2048, "f16"),    # 4 slices (100 rows), ragged last n-tile
    (128, 12288, 4096, "bf16"),  # more n-tiles than clusters fit: slices reduced by fp32 adds
])
def test_gemm_few_rows_split_k_matches_oracle(M, N, K, dtype):
    # at most 128 rows: K split into slices whose partials are summed on chip
    A = gen.normal16((9, 1), (M, K), 1.0, dtype)
    B = gen.normal16((9, 2), (K, N), 0.02, dtype)
    C = _out(M, N, dtype)
    nbytes = fx.flux_workspace_size(fx.FLUX_OP_GEMM, 1, M, N, K)
    assert nbytes >= M * N * 4  # the split form's fp32 rows
    ws = _ws(nbytes)
    for _ in range(2):
        fx.flux_gemm(M, N, K, DT[dtype], to_device(A, dtype), to_device(B, dtype), C, ws)
    _ok(ws)
    ref = oracle.gemm(oracle.widen(A, dtype), oracle.widen(B, dtype))
    check_close(oracle.widen(from_device(C), dtype), ref, f"few-row gemm {M}x{N}x{K} {dtype}")
    assert torch.count_nonzero(ws).item() == 0


def test_gemm_few_rows_split_k_integer_inputs_bit_exact():
    # |entries| <= 2, K = 1024: every partial and sum is an integer below 4097, exact in fp32
    # and (below 2048 in magnitude with high probability; checked) in fp16
    M, N, K = 128, 2048, 1024
    A = gen.integers16((10, 1), (M, K), -1, 1, "f16")
    B = gen.integers16((10, 2), (K, N), -1, 1, "f16")
    ref = oracle.gemm(oracle.widen(A, "f16"), oracle.widen(B, "f16"))
    assert np.abs(ref).max() <= 2048
    C = _out(M, N, "f16")
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM, 1, M, N, K))
    fx.flux_gemm(M, N, K, fx.FLUX_F16, to_device(A, "f16"), to_device(B, "f16"), C, ws)
    _ok(ws)
    assert np.array_equal(oracle.widen(from_device(C), "f16"), ref)


def test_gemm_k_zero_writes_zeros():
    C = _out(64, 64, "f16")
    a = torch.zeros(64, 8, dtype=torch.float16, device="cuda")
    fx.flux_gemm(64, 64, 0, fx.FLUX_F16, a, a, C, _ws(256))
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


# ---------------------------------------------------------------- AllGather + GEMM
def _ag_case(c, ready=None, opts=None):
    xs, ws_ = configs.ag_inputs(c)
    d = c.dtype
    X = [to_device(x, d) for x in xs]
    W = [to_device(w, d) for w in ws_]
    out = [_out(c.M, c.N // c.R, d) for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K))
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[d], X, W, out, ready, ws, opts=opts)
    return xs, ws_, out, ws


@pytest.mark.parametrize("R,M,N,K,dtype", [
    (1, 256, 512, 256, "f16"),
    (2, 256, 1024, 512, "f16"),
    (4, 512, 1024, 320, "bf16"),
    (8, 320, 576, 200, "f16"),     # 40 rows per shard (8-row boxes), ragged N and K tails
    (8, 1024, 2048, 128, "bf16"),  # shard = 128 rows: rank-rotated m order
    (16, 512, 2048, 256, "f16"),   # the most ranks a call takes: 32-row shards, 128 columns each
])
def test_ag_gemm_matches_oracle(R, M, N, K, dtype):
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=R, M=M, N=N, K=K, dtype=dtype, seed=20 + R)
    xs, w_s, out, ws = _ag_case(c)
    _ok(ws)
    ref = oracle.ag_gemm(xs, w_s, dtype)
    for r in range(R):
        check_close(oracle.widen(from_device(out[r]), dtype), ref[r], f"ag rank {r}")


def test_ag_gemm_flags_published_with_epoch():
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=4, M=512, N=1024, K=256, seed=31)
    flags = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    xs, w_s, out, ws = _ag_case(c, ready=flags, opts={"epoch": 7})
    _ok(ws)
    ref = oracle.ag_gemm(xs, w_s, c.dtype)
    for r in range(4):
        check_close(oracle.widen(from_device(out[r]), c.dtype), ref[r], f"ag flags rank {r}")


def test_ag_gemm_withheld_flag_times_out_and_gpu_stays_usable():
    # shard 2 never publishes: the pull of its rows must give up after the timeout
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=4, M=512, N=512, K=128, seed=32)
    flags = torch.tensor([1, 1, 0, 1], dtype=torch.int32, device="cuda")
    _, _, _, ws = _ag_case(c, ready=flags, opts={"timeout_ns": 20_000_000})
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_ERR_TIMEOUT
    assert rep["where"] == "ready flag" and rep["arg0"] == 2 and rep["arg1"] == 0
    # the same workspace (reset by flux_get_status) and GPU work normally afterwards
    flags.fill_(1)
    xs, w_s, out, ws = _ag_case(c, ready=flags)
    _ok(ws)
    ref = oracle.ag_gemm(xs, w_s, c.dtype)
    check_close(oracle.widen(from_device(out[2]), c.dtype), ref[2], "after timeout")


# ---------------------------------------------------------------- AllGather + GEMM, push form
@pytest.mark.parametrize("R,M,N,K,dtype,copiers", [
    (8, 320, 576, 200, "f16", 0),     # 40-row shards: blocks of 128 rows straddle shards
    (4, 512, 1024, 320, "bf16", 0),
    (8, 1024, 2048, 128, "bf16", 8),  # 8 copy CTAs, the others compute from the start
    (2, 256, 1024, 512, "f16", 1),    # one copy CTA
    (16, 512, 2048, 256, "f16", 0),   # the most ranks a call takes
])
def test_ag_gemm_push_form_matches_pull_and_oracle(R, M, N, K, dtype, copiers):
    # the push form: copy CTAs push every shard into one gathered copy (ready
    # count per 128-row block), tiles load A from it; same bits as the pull form
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=R, M=M, N=N, K=K, dtype=dtype, seed=120 + R)
    xs, w_s = configs.ag_inputs(c)
    X = [to_device(x, dtype) for x in xs]
    W = [to_device(w, dtype) for w in w_s]
    outs = {}
    for form in ("pull", "push"):
        out = [_out(M, N // R, dtype) for _ in range(R)]
        op = fx.FLUX_OP_AG_GEMM_PUSH if form == "push" else fx.FLUX_OP_AG_GEMM
        ws = _ws(fx.flux_workspace_size(op, R, M, N, K))
        opts = {"ag_push": 1, "moe_stage_ctas": copiers} if form == "push" else None
        flags = torch.ones(R, dtype=torch.int32, device="cuda")
        for _ in range(2):  # the second call finds the counters the first left at zero
            fx.flux_ag_gemm(R, M, N, K, DT[dtype], X, W, out, flags, ws, opts=opts)
        _ok(ws)
        outs[form] = out
    ref = oracle.ag_gemm(xs, w_s, dtype)
    for r in range(R):
        assert torch.equal(outs["pull"][r].view(torch.int16), outs["push"][r].view(torch.int16)), r
        check_close(oracle.widen(from_device(outs["push"][r]), dtype), ref[r], f"push ag rank {r}")


def test_ag_gemm_push_form_needs_its_workspace():
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=2, M=256, N=512, K=256, seed=126)
    xs, w_s = configs.ag_inputs(c)
    out = [_out(c.M, c.N // c.R, c.dtype) for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K))
    with pytest.raises(fx.FluxError, match="WORKSPACE"):
        fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], [to_device(x, c.dtype) for x in xs],
                        [to_device(w, c.dtype) for w in w_s], out, None, ws, opts={"ag_push": 1})


def test_ag_gemm_push_withheld_flag_times_out_and_gpu_stays_usable():
    # shard 1 never publishes: the push copy of its rows gives up after the
    # timeout, and so do the tiles waiting for those rows' blocks
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=4, M=512, N=512, K=128, seed=127)
    xs, w_s = configs.ag_inputs(c)
    X = [to_device(x, c.dtype) for x in xs]
    W = [to_device(w, c.dtype) for w in w_s]
    out = [_out(c.M, c.N // c.R, c.dtype) for _ in range(c.R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM_PUSH, c.R, c.M, c.N, c.K))
    flags = torch.tensor([1, 0, 1, 1], dtype=torch.int32, device="cuda")
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, flags, ws,
                    opts={"ag_push": 1, "timeout_ns": 20_000_000})
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_ERR_TIMEOUT
    flags.fill_(1)
    fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, flags, ws, opts={"ag_push": 1})
    _ok(ws)
    ref = oracle.ag_gemm(xs, w_s, c.dtype)
    for r in range(c.R):
        check_close(oracle.widen(from_device(out[r]), c.dtype), ref[r], f"push after timeout rank {r}")


# ---------------------------------------------------------------- GEMM + ReduceScatter
def _rs_case(c, opts=None, ws=None, calls=1):
    As, Bs = configs.rs_inputs(c)
    d = c.dtype
    A = [to_device(a, d) for a in As]
    B = [to_device(b, d) for b in Bs]
    out = [_out(c.M // c.R, c.N, d) for _ in range(c.R)]
    if ws is None:
        ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
    for _ in range(calls):
        fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[d], A, B, out, ws, opts=opts)
    return As, Bs, out, ws


def test_rs_config_r2_small_matches_oracle():
    c = configs.CONFIGS["rs_r2_small"]
    As, Bs, out, ws = _rs_case(c)
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for o in range(c.R):
        check_close(oracle.widen(from_device(out[o]), c.dtype), ref[o], f"rs owner {o}")


@pytest.mark.parametrize("R,M,N,K,dtype,num_ctas", [
    (2, 256, 512, 1024, "f16", 0),
    (4, 512, 1024, 1024, "bf16", 8),    # many units per CTA: strided whole-tile schedule
    (8, 192, 264, 576, "f16", 0),       # ragged M/N tails, 24-row owner chunks
    (8, 128, 2048, 4096, "bf16", 0),    # decode-like: split along K over the grid
    (8, 128, 2048, 4096, "bf16", 5),    # odd grid: k ranges straddle tiles
    (1, 300, 136, 200, "f16", 0),
    (16, 256, 512, 2048, "bf16", 0),    # the most ranks a call takes: 16-row owner chunks
    (16, 128, 1024, 8192, "bf16", 0),   # decode-like at 16 ranks: 8-row owner chunks, stream-K
])
def test_gemm_rs_matches_oracle(R, M, N, K, dtype, num_ctas):
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=R, M=M, N=N, K=K, dtype=dtype, seed=40 + R)
    opts = {"num_ctas": num_ctas} if num_ctas else None
    As, Bs, out, ws = _rs_case(c, opts=opts)
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"rs owner {o}")


def test_gemm_rs_integer_inputs_bit_exact_and_workspace_returns_to_zero():
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=4, M=256, N=512, K=128, dist="int", seed=45)
    As, Bs, out, ws = _rs_case(c, calls=3)  # repeated calls reuse the zeroed accumulators
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for o in range(c.R):
        assert np.array_equal(oracle.widen(from_device(out[o]), c.dtype), ref[o])
    assert torch.count_nonzero(ws).item() == 0


@pytest.mark.parametrize("R,M,N,K,dtype,num_ctas", [
    (4, 512, 1024, 1024, "bf16", 0),   # whole 512 x 512 cluster units
    (8, 128, 2048, 4096, "bf16", 0),   # decode-like shape: no k split in this mode
    (8, 192, 264, 576, "f16", 8),      # ragged tails on two clusters: a tile's ranks alternate
])
def test_gemm_rs_deterministic_repeats_bit_for_bit(R, M, N, K, dtype, num_ctas):
    # ranks add in ascending order: a second call on the re-zeroed workspace gives the same bits
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=R, M=M, N=N, K=K, dtype=dtype, seed=60 + R)
    opts = {"deterministic_rs": 1, "num_ctas": num_ctas}
    As, Bs, out, ws = _rs_case(c, opts=opts)
    _ok(ws)
    first = [o.clone() for o in out]
    fx.flux_gemm_rs(R, M, N, K, DT[dtype], [to_device(a, dtype) for a in As],
                    [to_device(b, dtype) for b in Bs], out, ws, opts=opts)
    _ok(ws)
    for o in range(R):
        assert torch.equal(first[o].view(torch.int16), out[o].view(torch.int16)), f"owner {o}"
    ref = oracle.gemm_rs(As, Bs, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"deterministic rs owner {o}")
    assert torch.count_nonzero(ws).item() == 0


def test_gemm_rs_deterministic_integer_inputs_bit_exact():
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=4, M=256, N=512, K=128, dist="int", seed=46)
    As, Bs, out, ws = _rs_case(c, opts={"deterministic_rs": 1})
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for o in range(c.R):
        assert np.array_equal(oracle.widen(from_device(out[o]), c.dtype), ref[o])


def test_gemm_rs_owner_chunk_layout_is_exact():
    # one-hot rows: each owner's chunk must hold exactly its rows (bit-exact layout)
    R, M, N, K = 4, 256, 256, 256
    Kr = K // R
    As = [np.zeros((M, Kr), np.float16) for _ in range(R)]
    Bs = [np.zeros((Kr, N), np.float16) for _ in range(R)]
    for r in range(R):
        for i in range(M):
            As[r][i, i % Kr] = 1.0
        for k in range(Kr):
            Bs[r][k, (k * 3 + r) % N] = float(r + 1)
    A = [to_device(a, "f16") for a in As]
    B = [to_device(b, "f16") for b in Bs]
    out = [_out(M // R, N, "f16") for _ in range(R)]
    ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, R, M, N, K))
    fx.flux_gemm_rs(R, M, N, K, fx.FLUX_F16, A, B, out, ws)
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, "f16")
    for o in range(R):
        assert np.array_equal(from_device(out[o]).astype(np.float64), ref[o])


# ---------------------------------------------------------------- argument checks (GPU present)
def test_argument_errors_launch_nothing():
    a = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    ws = _ws(256)
    with pytest.raises(fx.FluxError, match="INVALID_ARG"):
        fx.flux_ag_gemm(3, 64, 64, 64, fx.FLUX_F16, [a] * 3, [a] * 3, [a] * 3, None, ws)
    with pytest.raises(fx.FluxError, match="UNSUPPORTED"):
        fx.flux_gemm(64, 64, 60, fx.FLUX_F16, a, a, a, ws)
    with pytest.raises(fx.FluxError, match="WORKSPACE"):
        fx.flux_gemm_rs(2, 64, 64, 64, fx.FLUX_F16, [a] * 2, [a] * 2, [a] * 2, ws)
    with pytest.raises(fx.FluxError, match="UNSUPPORTED"):
        fx.flux_gemm(64, 64, 64, fx.FLUX_F16, a.data_ptr() + 2, a, a, ws)


# ---------------------------------------------------------------- unit schedules
def _static_ws_bytes(op, R, M, N, K):
    """Workspace without the dynamic schedule's mailboxes (the static schedule runs)."""
    if op == fx.FLUX_OP_AG_GEMM:
        return 256
    # header + arrival counters (4 per 128 x 256 tile) + fp32 owner rows
    return 256 + -(-((-(-M // 128)) * (-(-N // 256)) * 16) // 256) * 256 + M * N * 4


@pytest.mark.parametrize("num_ctas,N", [
    (0, 16384),   # 8 ranks x 4 m-units x 4 n-units = 128 units, the last 38 claimed as halves
    (8, 16384),   # two regions, 64+ units each; the last 2 units as halves
    (0, 6144),    # N/R = 768: every rank's last n-unit is 256 wide (its second half is empty)
    (0, 5120),    # N/R = 640: last n-units 128 wide
])
def test_ag_gemm_dynamic_schedule_matches_static_bit_for_bit(num_ctas, N):
    # the regions claim repeatedly; the last units of the schedule are split
    # into 256-column halves, halves past N are skipped
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=8, M=2048, N=N, K=256, dtype="bf16", seed=71)
    xs, w_s = configs.ag_inputs(c)
    X = [to_device(x, c.dtype) for x in xs]
    W = [to_device(w, c.dtype) for w in w_s]
    opts = {"num_ctas": num_ctas} if num_ctas else None
    outs = {}
    for name, nbytes in (("static", _static_ws_bytes(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K)),
                         ("dynamic", fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K))):
        ws = _ws(nbytes)
        out = [_out(c.M, c.N // c.R, c.dtype) for _ in range(c.R)]
        for _ in range(2):  # the second call runs on the schedule the first left zeroed
            fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, None, ws, opts=opts)
        _ok(ws)
        assert torch.count_nonzero(ws).item() == 0, name
        outs[name] = out
    for r in range(c.R):
        assert torch.equal(outs["static"][r].view(torch.int16), outs["dynamic"][r].view(torch.int16))
    ref = oracle.ag_gemm(xs, w_s, c.dtype)
    for r in (0, 5):
        check_close(oracle.widen(from_device(outs["dynamic"][r]), c.dtype), ref[r], f"ag dyn rank {r}")


@pytest.mark.parametrize("rs_tile", [1, 2, 3])
@pytest.mark.parametrize("num_ctas", [0, 12])
def test_gemm_rs_dynamic_schedule_integer_inputs_bit_exact(num_ctas, rs_tile):
    # integer inputs: every fp32 partial and sum is exact, whatever the order of the adds
    # (rs_tile 1: regions of 4 with 256 x 512 pair tiles; 2: regions of 8, 256 x 256;
    # 3: regions of 4, each claiming a tile and computing all its ranks' partials)
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=8, M=1024, N=4096, K=512, dist="int", seed=72)
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, c.dtype) for a in As]
    B = [to_device(b, c.dtype) for b in Bs]
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    opts = {"num_ctas": num_ctas, "rs_tile": rs_tile}
    for name, nbytes in (("static", _static_ws_bytes(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K)),
                         ("dynamic", fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))):
        ws = _ws(nbytes)
        out = [_out(c.M // c.R, c.N, c.dtype) for _ in range(c.R)]
        for _ in range(2):
            fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws, opts=opts)
        _ok(ws)
        for o in range(c.R):
            assert np.array_equal(oracle.widen(from_device(out[o]), c.dtype), ref[o]), (name, o)
        assert torch.count_nonzero(ws).item() == 0, name


@pytest.mark.parametrize("K", [128, 1024])
@pytest.mark.parametrize("form", ["dynamic", "static"])
def test_ag_gemm_accumulator_halves_match_whole_bit_for_bit(form, K):
    # 256 x 512 pair tiles hand their accumulator back in two halves (default)
    # or whole (acc_whole): the next tile's first k-slices (2 of them at
    # K = 128, the ring's 4 at K = 1024) run their first-half MMAs early; each
    # half still accumulates in k order, so the bits are those of the whole
    # hand-over.  N/R = 768: every rank's last tile is 256 wide (no early MMAs)
    c = configs.small(configs.CONFIGS["ag_mlp0"], R=8, M=1024, N=6144, K=K, dtype="f16", seed=73)
    xs, w_s = configs.ag_inputs(c)
    X = [to_device(x, c.dtype) for x in xs]
    W = [to_device(w, c.dtype) for w in w_s]
    nbytes = (_static_ws_bytes(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K) if form == "static"
              else fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, c.R, c.M, c.N, c.K))
    outs = []
    for whole in (0, 1):
        ws = _ws(nbytes)
        out = [_out(c.M, c.N // c.R, c.dtype) for _ in range(c.R)]
        fx.flux_ag_gemm(c.R, c.M, c.N, c.K, DT[c.dtype], X, W, out, None, ws, opts={"acc_whole": whole})
        _ok(ws)
        outs.append(out)
    for r in range(c.R):
        assert torch.equal(outs[0][r].view(torch.int16), outs[1][r].view(torch.int16)), f"rank {r}"
    ref = oracle.ag_gemm(xs, w_s, c.dtype)
    for r in (0, 7):
        check_close(oracle.widen(from_device(outs[0][r]), c.dtype), ref[r], f"ag halves rank {r}")


@pytest.mark.parametrize("N", [1288, 1280])
@pytest.mark.parametrize("rs_tile", [1, 3])
def test_gemm_rs_accumulator_halves_integer_inputs_bit_exact(rs_tile, N):
    # GEMM-RS's 256 x 512 pair tiles with the two-half hand-over (default) and
    # the whole one; integer inputs make every fp32 sum exact in any order.
    # N = 1288: the last tile's second half holds 8 columns; N = 1280: the
    # last tile is 256 wide.  K / R = 512: 8 k-slices per rank, twice the ring
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=8, M=1024, N=N, K=4096, dist="int", seed=74)
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, c.dtype) for a in As]
    B = [to_device(b, c.dtype) for b in Bs]
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for whole in (0, 1):
        ws = _ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K))
        out = [_out(c.M // c.R, c.N, c.dtype) for _ in range(c.R)]
        for _ in range(2):
            fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws,
                            opts={"rs_tile": rs_tile, "acc_whole": whole})
        _ok(ws)
        for o in range(c.R):
            assert np.array_equal(oracle.widen(from_device(out[o]), c.dtype), ref[o]), (whole, o)
        assert torch.count_nonzero(ws).item() == 0


@pytest.mark.parametrize("M", [1000, 1024])
@pytest.mark.parametrize("rs_group", [1, 2, 4, 8])
@pytest.mark.parametrize("num_ctas", [0, 12])
def test_gemm_rs_rank_groups_integer_inputs_bit_exact(rs_group, num_ctas, M):
    # a region sums the partials of rs_group ranks of one tile in TMEM and adds
    # the sum once; integer inputs make every sum exact in any order.  Groups
    # of all 8 ranks with 128-row owner chunks (M = 1024) store their sums
    # straight into the owners' 16-bit rows; the last groups, claimed rank by
    # rank, still go through the fp32 rows.  Two calls on one workspace: the
    # schedule and the counters are left clean
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=8, M=M, N=2056, K=8 * 1024, dist="int", seed=77)
    As, Bs = configs.rs_inputs(c)
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    opts = {"rs_group": rs_group}
    if num_ctas:
        opts["num_ctas"] = num_ctas
    _, _, out, ws = _rs_case(c, opts=opts, calls=2)
    _ok(ws)
    for o in range(c.R):
        assert np.array_equal(oracle.widen(from_device(out[o]), c.dtype), ref[o]), o
    assert torch.count_nonzero(ws).item() == 0


@pytest.mark.parametrize("R,M,N,K,dtype,rs_group", [
    (8, 1024, 2048, 8192, "bf16", 2),
    (4, 512, 1032, 4096, "f16", 4),    # ragged last n-unit (8 columns past 1024)
    (16, 1024, 2048, 4096, "f16", 2),  # the most ranks a call takes
    (6, 768, 1024, 3072, "bf16", 3),   # a group of 3 (6 ranks)
    (6, 768, 1024, 3072, "bf16", 4),   # 4 does not divide 6: each rank added on its own
    (8, 2048, 2056, 8192, "bf16", 8),  # all ranks in a group: sums stored as 16-bit, ragged N
    (16, 2048, 1024, 4096, "f16", 16), # all 16 ranks, 128-row owner chunks
])
def test_gemm_rs_rank_groups_match_oracle(R, M, N, K, dtype, rs_group):
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=R, M=M, N=N, K=K, dtype=dtype, seed=90 + R)
    As, Bs, out, ws = _rs_case(c, opts={"rs_group": rs_group})
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"rs group {rs_group} owner {o}")
    assert torch.count_nonzero(ws).item() == 0


@pytest.mark.parametrize("R,M,N,K,dtype,num_ctas", [
    (8, 1000, 2056, 1024, "f16", 16),   # ragged M and N tails, 125-row owner chunks
    (4, 512, 1032, 2048, "bf16", 16),   # ragged last n-unit (8 columns past 1024)
    (8, 2048, 4096, 4096, "bf16", 0),   # every SM: 8-CTA clusters where they fit, pairs elsewhere
    (16, 1024, 2048, 2048, "f16", 0),   # the most ranks a call takes
])
@pytest.mark.parametrize("rs_tile", [2, 3])
def test_gemm_rs_alternative_forms_match_oracle(R, M, N, K, dtype, num_ctas, rs_tile):
    # rs_tile 2: regions of 8 with 256 x 256 tiles; 3: tile-major regions of 4
    c = configs.small(configs.CONFIGS["rs_mlp1"], R=R, M=M, N=N, K=K, dtype=dtype, seed=80 + R)
    opts = {"rs_tile": rs_tile, "num_ctas": num_ctas}
    As, Bs, out, ws = _rs_case(c, opts=opts, calls=2)
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"rs form {rs_tile}, owner {o}")
    assert torch.count_nonzero(ws).item() == 0


# ---------------------------------------------------------------- cluster ReduceScatter (few rows)
@pytest.mark.parametrize("R,M,N,K,dtype", [
    (8, 128, 2048, 4096, "bf16"),   # decode-like: 8 n-tiles on 8 clusters, 2 partials per CTA
    (4, 128, 1000, 2048, "f16"),    # ragged last n-tile (1000 = 3 x 256 + 232)
    (8, 40, 264, 576, "f16"),       # 5 rows per owner, ragged k tail (72 per rank)
    (4, 64, 4096, 1024, "bf16"),    # 16 clusters, rows 64..127 of each tile empty
    (8, 16, 512, 256, "bf16"),      # 2 rows per owner, one k-slice per rank
])
def test_gemm_rs_cluster_form_matches_oracle(R, M, N, K, dtype):
    c = configs.small(configs.CONFIGS["rs_decode"], R=R, M=M, N=N, K=K, dtype=dtype, seed=90 + R)
    As, Bs, out, ws = _rs_case(c)
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, dtype)
    for o in range(R):
        check_close(oracle.widen(from_device(out[o]), dtype), ref[o], f"cluster rs owner {o}")


@pytest.mark.parametrize("R", [4, 8])
def test_gemm_rs_cluster_form_integer_inputs_bit_exact_and_repeatable(R):
    # exact fp32 partials and sums; the slot order is fixed, so repeat calls give the same bits
    # |entries| <= 2, 64 products per rank: every sum is an integer below 2049, exact in f16
    c = configs.small(configs.CONFIGS["rs_decode"], R=R, M=128, N=1536, K=R * 64, dist="int",
                      dtype="f16", seed=95 + R)
    As, Bs, out, ws = _rs_case(c, calls=2)
    _ok(ws)
    ref = oracle.gemm_rs(As, Bs, c.dtype)
    for o in range(R):
        assert np.array_equal(oracle.widen(from_device(out[o]), c.dtype), ref[o]), o
    first = [o.clone() for o in out]
    fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], [to_device(a, c.dtype) for a in As],
                    [to_device(b, c.dtype) for b in Bs], out, ws)
    _ok(ws)
    for o in range(R):
        assert torch.equal(first[o].view(torch.int16), out[o].view(torch.int16))
    assert torch.count_nonzero(ws).item() == 0


def test_launch_info_reports_the_dense_launch_shapes():
    # store mode: regions of 8 CTAs (8-CTA clusters preferred); reduce mode: regions of 4
    for op, cl in ((fx.FLUX_OP_AG_GEMM, 8), (fx.FLUX_OP_GEMM, 8), (fx.FLUX_OP_GEMM_RS, 4)):
        info = fx.flux_launch_info(op, fx.FLUX_F16)
        assert info["cluster_ctas"] == cl, (op, info)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert cl <= info["resident_ctas"] <= sms and info["resident_ctas"] % cl == 0, (op, info)
    with pytest.raises(fx.FluxError):
        fx.flux_launch_info(fx.FLUX_OP_MOE_AG, fx.FLUX_F16)
