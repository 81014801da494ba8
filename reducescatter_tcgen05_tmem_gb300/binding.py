"""ctypes binding of libflux_gb300.so: argument marshalling only.

Every function here has the name and the argument order of its C entry point
in ``include/flux_gb300.h``.  Pointer arguments accept torch tensors (their
``data_ptr()`` is passed), plain integers, or None for NULL; arrays of R
pointers accept a list of tensors.  ``stream`` defaults to torch's current
CUDA stream.  A non-OK status raises :class:`FluxError`.  No step of the
computation happens in Python, and there is no fallback: importing this module
raises if the compiled library is missing.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# FLUX_CHECKED=1 in the environment loads the checked build (bounds checks in
# every kernel, see flux_checks_enabled in the header) instead of the regular one
CHECKED = os.environ.get("FLUX_CHECKED", "") not in ("", "0")
LIB_PATH = os.path.join(HERE, "libflux_gb300_checked.so" if CHECKED else "libflux_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m reducescatter_tcgen05_tmem_gb300.build` "
        "(the library has no CPU or Python fallback)")

_lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------- constants
FLUX_OK = 0
FLUX_ERR_INVALID_ARG = 1
FLUX_ERR_UNSUPPORTED = 2
FLUX_ERR_WORKSPACE = 3
FLUX_ERR_CUDA = 4
FLUX_ERR_TIMEOUT = 5
FLUX_ERR_NO_DEVICE = 6

FLUX_F16 = 0
FLUX_BF16 = 1

FLUX_OP_GEMM = 0
FLUX_OP_AG_GEMM = 1
FLUX_OP_GEMM_RS = 2
FLUX_OP_MOE_AG = 3
FLUX_OP_MOE_RS = 4
FLUX_OP_MLP = 5
FLUX_OP_MOE_LAYERS = 6
FLUX_OP_MOE_EP_AG = 7
FLUX_OP_MOE_EP_RS = 8
FLUX_OP_AG_GEMM_PUSH = 9

FLUX_MAX_RANKS = 16
FLUX_MAX_EXPERTS = 1024
FLUX_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

WAIT_SITES = {1: "ready flag", 2: "smem slot free", 3: "smem slot full",
              4: "accumulator free", 5: "accumulator full", 6: "drain",
              7: "deterministic turn", 8: "staged rows", 9: "unit schedule",
              10: "cluster shape", 11: "grid barrier", 12: "cluster exchange", 13: "check"}


class flux_opts_t(ctypes.Structure):
    _fields_ = [("epoch", ctypes.c_uint32), ("reserved0", ctypes.c_uint32),
                ("timeout_ns", ctypes.c_uint64), ("num_ctas", ctypes.c_int32),
                ("group_n", ctypes.c_int32), ("tiles_per_group", ctypes.c_int32),
                ("deterministic_rs", ctypes.c_int32), ("moe_pull_gather", ctypes.c_int32),
                ("moe_stage_ctas", ctypes.c_int32), ("rs_tile", ctypes.c_int32),
                ("moe_l1_ranks", ctypes.c_int32), ("trace", ctypes.c_void_p),
                ("trace_words", ctypes.c_uint64), ("ag_push", ctypes.c_int32),
                ("debug_probe", ctypes.c_int32),
                ("moe_static_schedule", ctypes.c_int32), ("rs_group", ctypes.c_int32),
                ("acc_whole", ctypes.c_int32)]


class flux_device_report_t(ctypes.Structure):
    _fields_ = [("status", ctypes.c_uint32), ("where", ctypes.c_uint32),
                ("arg0", ctypes.c_uint32), ("arg1", ctypes.c_uint32)]


class FluxError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = _lib.flux_status_string(status).decode()
        extra = ""
        if status == FLUX_ERR_CUDA:
            extra = f" (cudaError {_lib.flux_last_cuda_error()})"
        super().__init__(f"{what}: {name}{extra}")


_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_vpp = ctypes.POINTER(ctypes.c_void_p)
_opt = ctypes.POINTER(flux_opts_t)

_SIGS = {
    "flux_version": ([], ctypes.c_int),
    "flux_checks_enabled": ([], ctypes.c_int),
    "flux_opts_size": ([], _sz),
    "flux_status_string": ([_i], ctypes.c_char_p),
    "flux_last_cuda_error": ([], ctypes.c_int),
    "flux_workspace_size": ([_i, _i, _i, _i, _i], _sz),
    "flux_moe_workspace_size": ([_i, _i, _i, _i, _i, _i, _i], _sz),
    "flux_workspace_init": ([_vp, _sz, _vp], _i),
    "flux_get_status": ([_vp, _sz, _vp, ctypes.POINTER(flux_device_report_t)], _i),
    "flux_gemm": ([_i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _opt, _vp], _i),
    "flux_ag_gemm": ([_i, _i, _i, _i, _i, _vpp, _vpp, _vpp, _vp, _vp, _sz, _opt, _vp], _i),
    "flux_gemm_rs": ([_i, _i, _i, _i, _i, _vpp, _vpp, _vpp, _vp, _sz, _opt, _vp], _i),
    "flux_gemm_rs_noalloc": ([_i, _i, _i, _i, _i, _vpp, _vpp, _vpp, _opt, _vp], _i),
    "flux_moe_topk_gate": ([_i, _i, _i, _vp, _vp, _vp, _vp], _i),
    "flux_moe_route": ([_i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i),
    "flux_moe_ag_grouped_gemm": ([_i, _i, _i, _i, _i, _i, _i, _vpp, _vpp, _vp, _vpp, _vp, _vp,
                                  _vp, _vp, _vp, _vp, _sz, _opt, _vp], _i),
    "flux_moe_grouped_gemm_rs": ([_i, _i, _i, _i, _i, _i, _i, _vpp, _vpp, _vp, _vp, _vp, _vp,
                                  _vp, _vpp, _vp, _sz, _opt, _vp], _i),
    "flux_mlp_ag_rs": ([_i, _i, _i, _i, _i, _vpp, _vpp, _vpp, _vpp, _vpp, _vp, _vp, _sz, _opt, _vp], _i),
    "flux_moe_layers": ([_i, _i, _i, _i, _i, _i, _i, _vpp, _vpp, _vpp, _vp, _vp, _vpp, _vpp, _vp,
                         _vp, _sz, _opt, _vp], _i),
    "flux_tune_ag_gemm": ([_i, _i, _i, _i, _i, _vpp, _vpp, _vpp, _vp, _vp, _sz, _vp, _opt], _i),
    "flux_tune_gemm_rs": ([_i, _i, _i, _i, _i, _vpp, _vpp, _vpp, _vp, _sz, _vp, _opt], _i),
    "flux_tune_moe_layer0": ([_i, _i, _i, _i, _i, _i, _i, _i, _vpp, _vpp, _vp, _vpp, _vp, _vp,
                              _vp, _vp, _vp, _vp, _sz, _vp, _opt], _i),
    "flux_tune_moe_layer1": ([_i, _i, _i, _i, _i, _i, _i, _i, _vpp, _vpp, _vp, _vp, _vp, _vp,
                              _vp, _vpp, _vp, _sz, _vp, _opt], _i),
    "flux_launch_info": ([_i, _i, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)], _i),
    "flux_tune_clear": ([], None),
    "flux_tune_count": ([], _i),
    "flux_moe_ep_dispatch_gemm": ([_i, _i, _i, _i, _i, _i, _i, _i, _vpp, _vpp, _vp, _vpp, _vp,
                                   _vp, _vp, _vp, _vp, _vp, _sz, _opt, _vp], _i),
    "flux_moe_ep_gemm_combine": ([_i, _i, _i, _i, _i, _i, _i, _i, _vpp, _vpp, _vp, _vp, _vp,
                                  _vp, _vp, _vpp, _vp, _sz, _opt, _vp], _i),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

EXPORTED = tuple(_SIGS)
if _lib.flux_opts_size() != ctypes.sizeof(flux_opts_t):
    raise ImportError(f"flux_opts_t: the binding's copy ({ctypes.sizeof(flux_opts_t)} bytes) does not match "
                      f"{LIB_PATH} ({_lib.flux_opts_size()} bytes); rebuild the library")
_OPT_FIELDS = frozenset(name for name, _ in flux_opts_t._fields_)


# ---------------------------------------------------------------- marshalling
def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptrs(xs):
    arr = (ctypes.c_void_p * len(xs))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def _nbytes(t):
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _opts(opts):
    if opts is None:
        return None
    if isinstance(opts, dict):
        o = flux_opts_t()
        for k, v in opts.items():
            if k not in _OPT_FIELDS:
                raise KeyError(f"flux_opts_t has no field {k!r}")
            if k == "trace" and v is not None and not isinstance(v, int):
                # a tensor: its address, and its size unless given
                if "trace_words" not in opts:
                    o.trace_words = _nbytes(v) // 8
                v = v.data_ptr()
            setattr(o, k, v)
        opts = o
    return ctypes.byref(opts)


def _check(st, what):
    if st != FLUX_OK:
        raise FluxError(st, what)


def dtype_code(t) -> int:
    """FLUX_F16 / FLUX_BF16 for a torch dtype or tensor."""
    import torch
    dt = t.dtype if hasattr(t, "dtype") else t
    if dt == torch.float16:
        return FLUX_F16
    if dt == torch.bfloat16:
        return FLUX_BF16
    raise ValueError(f"unsupported dtype {dt}")


# ---------------------------------------------------------------- API (same names as the C ABI)
def flux_version() -> int:
    return _lib.flux_version()


def flux_checks_enabled() -> bool:
    return bool(_lib.flux_checks_enabled())


def flux_opts_size() -> int:
    return int(_lib.flux_opts_size())


def flux_status_string(status: int) -> str:
    return _lib.flux_status_string(status).decode()


def flux_workspace_size(op: int, R: int, M: int, N: int, K: int) -> int:
    return int(_lib.flux_workspace_size(op, R, M, N, K))


def flux_moe_workspace_size(op: int, R: int, T: int, H: int, F: int, E: int, topk: int) -> int:
    return int(_lib.flux_moe_workspace_size(op, R, T, H, F, E, topk))


def flux_workspace_init(workspace, stream=None) -> None:
    _check(_lib.flux_workspace_init(_ptr(workspace), _nbytes(workspace), _stream(stream)),
           "flux_workspace_init")


def flux_get_status(workspace, stream=None):
    """(status, report) after synchronising the stream; never raises for device errors."""
    rep = flux_device_report_t()
    st = _lib.flux_get_status(_ptr(workspace), _nbytes(workspace), _stream(stream), ctypes.byref(rep))
    if st in (FLUX_ERR_CUDA, FLUX_ERR_WORKSPACE):
        raise FluxError(st, "flux_get_status")
    return st, {"status": rep.status, "where": WAIT_SITES.get(rep.where, rep.where),
                "arg0": rep.arg0, "arg1": rep.arg1}


def flux_gemm(M, N, K, dtype, A, B, C, workspace, opts=None, stream=None) -> None:
    _check(_lib.flux_gemm(M, N, K, dtype, _ptr(A), _ptr(B), _ptr(C), _ptr(workspace),
                          _nbytes(workspace), _opts(opts), _stream(stream)), "flux_gemm")


def flux_ag_gemm(R, M, N, K, dtype, x_shards, w_shards, out, ready_flags, workspace,
                 opts=None, stream=None) -> None:
    _check(_lib.flux_ag_gemm(R, M, N, K, dtype, _ptrs(x_shards), _ptrs(w_shards), _ptrs(out),
                             _ptr(ready_flags), _ptr(workspace), _nbytes(workspace), _opts(opts),
                             _stream(stream)), "flux_ag_gemm")


def flux_gemm_rs(R, M, N, K, dtype, a_shards, b_shards, out, workspace, opts=None,
                 stream=None) -> None:
    _check(_lib.flux_gemm_rs(R, M, N, K, dtype, _ptrs(a_shards), _ptrs(b_shards), _ptrs(out),
                             _ptr(workspace), _nbytes(workspace), _opts(opts), _stream(stream)),
           "flux_gemm_rs")


def flux_gemm_rs_noalloc(R, M, N, K, dtype, a_shards, b_shards, out, opts=None,
                         stream=None) -> None:
    """flux_gemm_rs without a workspace: scratch lives in a fixed device array of
    the library (FLUX_NOALLOC_SCRATCH_BYTES), for callers that cannot allocate."""
    _check(_lib.flux_gemm_rs_noalloc(R, M, N, K, dtype, _ptrs(a_shards), _ptrs(b_shards),
                                     _ptrs(out), _opts(opts), _stream(stream)),
           "flux_gemm_rs_noalloc")


def flux_moe_topk_gate(T, E, topk, logits, topk_ids, topk_weights, stream=None) -> None:
    """Top-k expert ids and softmax gate weights from fp32 router scores."""
    _check(_lib.flux_moe_topk_gate(T, E, topk, _ptr(logits), _ptr(topk_ids), _ptr(topk_weights),
                                   _stream(stream)), "flux_moe_topk_gate")


def flux_moe_route(T, E, topk, topk_ids, counts, offsets, slot_to_row, row_to_slot,
                   workspace=None, stream=None) -> None:
    _check(_lib.flux_moe_route(T, E, topk, _ptr(topk_ids), _ptr(counts), _ptr(offsets),
                               _ptr(slot_to_row), _ptr(row_to_slot), _ptr(workspace),
                               0 if workspace is None else _nbytes(workspace), _stream(stream)),
           "flux_moe_route")


def flux_moe_ag_grouped_gemm(R, T, H, F, E, topk, dtype, x_shards, w1_shards, topk_ids, h_out,
                             counts, offsets, slot_to_row, row_to_slot, ready_flags, workspace,
                             opts=None, stream=None) -> None:
    _check(_lib.flux_moe_ag_grouped_gemm(
        R, T, H, F, E, topk, dtype, _ptrs(x_shards), _ptrs(w1_shards), _ptr(topk_ids),
        _ptrs(h_out), _ptr(counts), _ptr(offsets), _ptr(slot_to_row), _ptr(row_to_slot),
        _ptr(ready_flags), _ptr(workspace), _nbytes(workspace), _opts(opts), _stream(stream)),
        "flux_moe_ag_grouped_gemm")


def flux_moe_grouped_gemm_rs(R, T, H, F, E, topk, dtype, h_shards, w2_shards, topk_ids,
                             topk_weights, offsets, slot_to_row, row_to_slot, out, workspace,
                             opts=None, stream=None) -> None:
    _check(_lib.flux_moe_grouped_gemm_rs(
        R, T, H, F, E, topk, dtype, _ptrs(h_shards), _ptrs(w2_shards), _ptr(topk_ids),
        _ptr(topk_weights), _ptr(offsets), _ptr(slot_to_row), _ptr(row_to_slot), _ptrs(out),
        _ptr(workspace), _nbytes(workspace), _opts(opts), _stream(stream)),
        "flux_moe_grouped_gemm_rs")


def flux_mlp_ag_rs(R, M, H, F, dtype, x_shards, w1_shards, h, w2_shards, out, ready_flags,
                   workspace, opts=None, stream=None) -> None:
    """The dense MLP in one call: h = AG-GEMM(X, W1), out = GEMM-RS(h, W2)."""
    _check(_lib.flux_mlp_ag_rs(R, M, H, F, dtype, _ptrs(x_shards), _ptrs(w1_shards), _ptrs(h),
                               _ptrs(w2_shards), _ptrs(out), _ptr(ready_flags), _ptr(workspace),
                               _nbytes(workspace), _opts(opts), _stream(stream)), "flux_mlp_ag_rs")


def flux_moe_layers(R, T, H, F, E, topk, dtype, x_shards, w1_shards, w2_shards, topk_ids,
                    topk_weights, h, out, ready_flags, workspace, opts=None, stream=None) -> None:
    """The MoE layer in one call: routing, layer0 into h, layer1 into out."""
    _check(_lib.flux_moe_layers(R, T, H, F, E, topk, dtype, _ptrs(x_shards), _ptrs(w1_shards),
                                _ptrs(w2_shards), _ptr(topk_ids), _ptr(topk_weights), _ptrs(h),
                                _ptrs(out), _ptr(ready_flags), _ptr(workspace), _nbytes(workspace),
                                _opts(opts), _stream(stream)), "flux_moe_layers")


def flux_moe_ep_dispatch_gemm(R, tp, T, H, F, E, topk, dtype, x_shards, w1_shards, topk_ids,
                              h_out, counts, offsets, slot_to_row, row_to_slot, ready_flags,
                              workspace, opts=None, stream=None) -> None:
    """MoE layer0 under an EP x TP split (tp ranks per expert group)."""
    _check(_lib.flux_moe_ep_dispatch_gemm(
        R, tp, T, H, F, E, topk, dtype, _ptrs(x_shards), _ptrs(w1_shards), _ptr(topk_ids),
        _ptrs(h_out), _ptr(counts), _ptr(offsets), _ptr(slot_to_row), _ptr(row_to_slot),
        _ptr(ready_flags), _ptr(workspace), _nbytes(workspace), _opts(opts), _stream(stream)),
        "flux_moe_ep_dispatch_gemm")


def flux_moe_ep_gemm_combine(R, tp, T, H, F, E, topk, dtype, h_shards, w2_shards, topk_ids,
                             topk_weights, offsets, slot_to_row, row_to_slot, out, workspace,
                             opts=None, stream=None) -> None:
    """MoE layer1 + top-k combine under an EP x TP split."""
    _check(_lib.flux_moe_ep_gemm_combine(
        R, tp, T, H, F, E, topk, dtype, _ptrs(h_shards), _ptrs(w2_shards), _ptr(topk_ids),
        _ptr(topk_weights), _ptr(offsets), _ptr(slot_to_row), _ptr(row_to_slot), _ptrs(out),
        _ptr(workspace), _nbytes(workspace), _opts(opts), _stream(stream)),
        "flux_moe_ep_gemm_combine")


def _tuned(st, what, best):
    _check(st, what)
    return {f: getattr(best, f) for f, _ in flux_opts_t._fields_}


def flux_tune_ag_gemm(R, M, N, K, dtype, x_shards, w_shards, out, ready_flags, workspace,
                      stream=None) -> dict:
    """Time the AllGather + GEMM candidates; record and return the fastest options."""
    best = flux_opts_t()
    return _tuned(_lib.flux_tune_ag_gemm(R, M, N, K, dtype, _ptrs(x_shards), _ptrs(w_shards),
                                         _ptrs(out), _ptr(ready_flags), _ptr(workspace),
                                         _nbytes(workspace), _stream(stream), ctypes.byref(best)),
                  "flux_tune_ag_gemm", best)


def flux_tune_gemm_rs(R, M, N, K, dtype, a_shards, b_shards, out, workspace, stream=None) -> dict:
    """Time the GEMM + ReduceScatter candidates; record and return the fastest options."""
    best = flux_opts_t()
    return _tuned(_lib.flux_tune_gemm_rs(R, M, N, K, dtype, _ptrs(a_shards), _ptrs(b_shards),
                                         _ptrs(out), _ptr(workspace), _nbytes(workspace),
                                         _stream(stream), ctypes.byref(best)),
                  "flux_tune_gemm_rs", best)


def flux_tune_moe_layer0(R, tp, T, H, F, E, topk, dtype, x_shards, w1_shards, topk_ids, h_out,
                         counts, offsets, slot_to_row, row_to_slot, ready_flags, workspace,
                         stream=None) -> dict:
    """Time the MoE layer0 candidates (staged / pull); record and return the fastest."""
    best = flux_opts_t()
    return _tuned(_lib.flux_tune_moe_layer0(
        R, tp, T, H, F, E, topk, dtype, _ptrs(x_shards), _ptrs(w1_shards), _ptr(topk_ids),
        _ptrs(h_out), _ptr(counts), _ptr(offsets), _ptr(slot_to_row), _ptr(row_to_slot),
        _ptr(ready_flags), _ptr(workspace), _nbytes(workspace), _stream(stream),
        ctypes.byref(best)), "flux_tune_moe_layer0", best)


def flux_tune_moe_layer1(R, tp, T, H, F, E, topk, dtype, h_shards, w2_shards, topk_ids,
                         topk_weights, offsets, slot_to_row, row_to_slot, out, workspace,
                         stream=None) -> dict:
    """Time the MoE layer1 candidates; record and return the fastest."""
    best = flux_opts_t()
    return _tuned(_lib.flux_tune_moe_layer1(
        R, tp, T, H, F, E, topk, dtype, _ptrs(h_shards), _ptrs(w2_shards), _ptr(topk_ids),
        _ptr(topk_weights), _ptr(offsets), _ptr(slot_to_row), _ptr(row_to_slot), _ptrs(out),
        _ptr(workspace), _nbytes(workspace), _stream(stream), ctypes.byref(best)),
        "flux_tune_moe_layer1", best)


def flux_tune_clear() -> None:
    _lib.flux_tune_clear()


def flux_tune_count() -> int:
    return _lib.flux_tune_count()


def flux_launch_info(op, dtype) -> dict:
    """CTAs per cluster and resident CTAs of a dense op's kernel on this GPU."""
    cl, res = ctypes.c_int(0), ctypes.c_int(0)
    _check(_lib.flux_launch_info(op, dtype, ctypes.byref(cl), ctypes.byref(res)), "flux_launch_info")
    return {"cluster_ctas": cl.value, "resident_ctas": res.value}
