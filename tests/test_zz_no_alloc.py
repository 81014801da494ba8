"""GEMM + ReduceScatter without a workspace (flux_gemm_rs_noalloc).

This entry point is for callers that cannot allocate device memory or pass a
workspace: plugin hosts and inference runtimes whose device-memory budget is
fixed before serving starts, and thin wrappers with no allocator of their own.
Its scratch is a fixed array inside the library.  The test calls it through
the C ABI twice in a row (the second call reuses the array the first one
left behind) and checks each result against the existing entry point,
flux_gemm_rs with a caller-provided workspace, within the parity tolerance.
It runs last in the suite and also passes on its own in a fresh process.
"""
import pytest

from tests.parity import check_close
from workloads import configs
from workloads.torch_io import to_device, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reducescatter_tcgen05_tmem_gb300 as fx  # noqa: E402

DT = {"f16": fx.FLUX_F16, "bf16": fx.FLUX_BF16}


def _reference(c, A, B):
    """The existing entry point with a caller-allocated workspace."""
    out = [torch.empty(c.M // c.R, c.N, dtype=torch_dtype(c.dtype), device="cuda") for _ in range(c.R)]
    ws = torch.zeros(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, c.R, c.M, c.N, c.K) // 4,
                     dtype=torch.int32, device="cuda")
    fx.flux_gemm_rs(c.R, c.M, c.N, c.K, DT[c.dtype], A, B, out, ws)
    st, rep = fx.flux_get_status(ws)
    assert st == fx.FLUX_OK, rep
    return out


@pytest.mark.parametrize("R,M,N,K,dtype", [
    (2, 128, 256, 512, "f16"),      # the R=2 GEMM+ReduceScatter workload
    (8, 128, 2048, 8192, "bf16"),   # decode-shaped: split along K, 1 MiB of fp32 accumulators
    (4, 192, 520, 1024, "f16"),     # ragged tiles
])
def test_noalloc_matches_workspace_entry_point_twice(R, M, N, K, dtype):
    c = configs.small(configs.CONFIGS["rs_r2_small"], R=R, M=M, N=N, K=K, dtype=dtype, seed=900 + R)
    As, Bs = configs.rs_inputs(c)
    A = [to_device(a, dtype) for a in As]
    B = [to_device(b, dtype) for b in Bs]
    ref = _reference(c, A, B)
    for call in range(2):
        out = [torch.full((M // R, N), float("nan"), dtype=torch_dtype(dtype), device="cuda")
               for _ in range(R)]
        fx.flux_gemm_rs_noalloc(R, M, N, K, DT[dtype], A, B, out)
        torch.cuda.synchronize()
        for o in range(R):
            check_close(out[o].double().cpu().numpy(), ref[o].double().cpu().numpy(),
                        f"call {call} owner {o}")


def test_noalloc_rejects_problems_larger_than_its_scratch():
    # 4096 x 12288 fp32 accumulators alone are 192 MiB > 16 MiB of built-in scratch
    need = fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, 8, 4096, 12288, 49152)
    assert need > fx.FLUX_NOALLOC_SCRATCH_BYTES
    a = torch.zeros(16, dtype=torch.float16, device="cuda")
    with pytest.raises(fx.FluxError, match="WORKSPACE"):
        fx.flux_gemm_rs_noalloc(8, 4096, 12288, 49152, fx.FLUX_F16, [a] * 8, [a] * 8, [a] * 8)
