"""GEMM + ReduceScatter without a workspace (flux_gemm_rs_noalloc).

This entry point is for callers that cannot allocate device memory or pass a
workspace: plugin hosts and inference runtimes whose device-memory budget is
fixed before serving starts, and thin wrappers with no allocator of their own.
Its scratch is a fixed array inside the library.  The tests call it through
the C ABI twice in a row (the second call reuses the array the first one
left behind) and check each result against the existing entry point,
flux_gemm_rs with a caller-provided workspace, and against the oracle, both
within the parity tolerance.  The file runs last in the suite and also
passes on its own in a fresh process.
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


def _problem(R, M, N, K, dtype, seed):
    c = configs.small(configs.CONFIGS["rs_r2_small"], R=R, M=M, N=N, K=K, dtype=dtype, seed=seed)
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, dtype) for a in As]
    B = [to_device(b, dtype) for b in Bs]
    return c, As, Bs, A, B


def _nan_outputs(c):
    return [torch.full((c.M // c.R, c.N), float("nan"), dtype=torch_dtype(c.dtype), device="cuda")
            for _ in range(c.R)]


def _reference(c, A, B, opts=None):
    """The existing entry point with a caller-allocated workspace."""
    out = _nan_outputs(c)
    ws = torch.zeros(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K) // 4,
                     dtype=torch.int32, device="cuda")
    fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws, opts)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    return out


def _check(c, As, Bs, got, ref, what):
    want = oracle.gemm_rs(As, Bs, c.dtype)
    for o in range(c.R):
        g = oracle.widen(from_device(got[o]), c.dtype)
        check_close(g, oracle.widen(from_device(ref[o]), c.dtype), f"{what} owner {o} vs flux_gemm_rs")
        check_close(g, want[o], f"{what} owner {o} vs oracle")


@pytest.mark.parametrize("R,M,N,K,dtype", [
    (2, 128, 256, 512, "f16"),      # the R=2 GEMM+ReduceScatter workload
    (8, 128, 2048, 8192, "bf16"),   # decode-shaped: the cluster form (no fp32 scratch rows)
    (8, 256, 2048, 8192, "bf16"),   # 256 rows: fp32 rows in the scratch, split along K
    (4, 192, 520, 1024, "f16"),     # ragged tiles
])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(R, M, N, K, dtype):
    c, As, Bs, A, B = _problem(R, M, N, K, dtype, 900 + R + M)
    ref = _reference(c, A, B)
    for call in range(2):
        out = _nan_outputs(c)
        fx.flux_gemm_rs_noalloc(R, M, N, K, DT[dtype], A, B, out)
        torch.cuda.synchronize()
        _check(c, As, Bs, out, ref, f"call {call}")


def test_noalloc_deterministic_after_a_larger_call_of_another_shape():
    # a larger call first leaves the shared scratch as it ends; a smaller call
    # in deterministic mode (its own static, whole-tile schedule) must then
    # start from a clean scratch and give the same bits as flux_gemm_rs in the
    # same mode with a workspace of its own
    big, As0, Bs0, A0, B0 = _problem(8, 512, 4096, 4096, "bf16", 971)
    out0 = _nan_outputs(big)
    fx.flux_gemm_rs_noalloc(big.R, big.M, big.N, big.K, DT[big.dtype], A0, B0, out0)
    c, As, Bs, A, B = _problem(4, 192, 520, 1024, "f16", 972)
    det = {"deterministic_rs": 1}
    ref = _reference(c, A, B, det)
    for call in range(2):
        out = _nan_outputs(c)
        fx.flux_gemm_rs_noalloc(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, det)
        torch.cuda.synchronize()
        for o in range(c.R):
            assert torch.equal(out[o], ref[o]), f"call {call} owner {o}: not the same bits"
        _check(c, As, Bs, out, ref, f"deterministic call {call}")
    _check(big, As0, Bs0, out0, _reference(big, A0, B0), "larger call")


def test_noalloc_refused_call_then_a_valid_one():
    c, As, Bs, A, B = _problem(2, 128, 256, 512, "f16", 973)
    bad = [torch.empty(c.M // c.R * c.N + 1, dtype=torch.float16, device="cuda")[1:].view(c.M // c.R, c.N)
           for _ in range(c.R)]  # 2-byte offset: not 16-byte aligned
    with pytest.raises(fx.FluxError, match="UNSUPPORTED"):
        fx.flux_gemm_rs_noalloc(c.R, c.M, c.N, c.K, fx.FLUX_F16, A, B, bad)
    out = _nan_outputs(c)
    fx.flux_gemm_rs_noalloc(c.R, c.M, c.N, c.K, fx.FLUX_F16, A, B, out)
    torch.cuda.synchronize()
    _check(c, As, Bs, out, _reference(c, A, B), "after a refused call")
    assert np.isfinite(oracle.widen(from_device(out[0]), "f16")).all()


def test_noalloc_rejects_problems_larger_than_its_scratch():
    # 4096 x 12288 fp32 accumulators alone are 192 MiB > 16 MiB of built-in scratch
    need = fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, 8, 4096, 12288, 49152)
    assert need > fx.FLUX_NOALLOC_SCRATCH_BYTES
    a = torch.zeros(16, dtype=torch.float16, device="cuda")
    with pytest.raises(fx.FluxError, match="WORKSPACE"):
        fx.flux_gemm_rs_noalloc(8, 4096, 12288, 49152, fx.FLUX_F16, [a] * 8, [a] * 8, [a] * 8)
