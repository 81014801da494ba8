"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before touching the GPU (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flux_gb300.h")


@pytest.fixture(scope="module")
def fx():
    from tests.conftest import ensure_built
    ensure_built()
    import reducescatter_tcgen05_tmem_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flux_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for want in ("flux_gemm", "flux_ag_gemm", "flux_gemm_rs", "flux_moe_route",
                 "flux_moe_ag_grouped_gemm", "flux_moe_grouped_gemm_rs", "flux_get_status"):
        assert want in names


def test_library_exports_every_declared_symbol(fx):
    lib = ctypes.CDLL(fx.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert name in fx.EXPORTED, f"{name} has no Python binding"


def _opts_fields_in_header():
    text = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} flux_opts_t;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    return re.findall(r"^\s*[a-z0-9_]+\*?\s+\*?([a-z0-9_]+);", body, flags=re.M)


def test_opts_struct_matches_the_header(fx):
    # the binding's copy of flux_opts_t has the header's fields in the header's
    # order and the size the library was compiled with
    names = [n for n, _ in fx.binding.flux_opts_t._fields_]
    assert names == _opts_fields_in_header()
    assert fx.flux_opts_size() == ctypes.sizeof(fx.binding.flux_opts_t)


class _WS:  # stand-in workspace: only its address and size are looked at
    def __init__(self, n, addr=1 << 20):
        self.n, self.addr = n, addr

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.n

    def element_size(self):
        return 1


def test_unknown_option_is_refused_before_the_call(fx):
    # a misspelt option name is an error, not a silently ignored attribute
    with pytest.raises(KeyError, match="acc_whol"):
        fx.flux_gemm(64, 64, 64, fx.FLUX_F16, FAKE, FAKE, FAKE, _WS(256), opts={"acc_whol": 1}, stream=0)


def test_version_and_status_strings(fx):
    assert fx.flux_version() >= 100
    assert fx.flux_status_string(fx.FLUX_ERR_TIMEOUT) == "FLUX_ERR_TIMEOUT"
    assert fx.flux_status_string(99) == "FLUX_ERR_UNKNOWN"


def _sched(units):
    # mailboxes of the dynamic unit schedule: (2 U + 6 x 64 regions) uint32, 256-byte rounded
    return -(-(2 * units + 384) * 4 // 256) * 256


def test_workspace_sizes(fx):
    # header + schedule of the 512 x 512 units (8 m-units x 24 n-units)
    assert fx.flux_workspace_size(fx.FLUX_OP_GEMM, 1, 4096, 12288, 6144) == 256 + _sched(8 * 24)
    # 8 ranks x 8 m-units x 12 n-units of 6144 columns
    assert fx.flux_workspace_size(fx.FLUX_OP_AG_GEMM, 8, 4096, 49152, 12288) == 256 + _sched(768)
    # header + counters (32 x 48 tiles x 4 quarters x 4 B) + fp32 owner chunks (M x N)
    # + schedule (8 ranks x 8 x 24 units)
    rs = 256 + 32 * 48 * 16 + 4096 * 12288 * 4 + _sched(8 * 8 * 24)
    assert fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, 8, 4096, 12288, 49152) == rs
    # the MLP's workspace serves both of its calls
    assert fx.flux_workspace_size(fx.FLUX_OP_MLP, 8, 4096, 12288, 49152) == rs
    assert fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, 0, 1, 1, 1) == 0
    assert fx.flux_workspace_size(99, 1, 1, 1, 1) == 0
    s = fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, 8, 4096, 4096, 14336, 8, 2)
    # layer1: header, tile table, routing (counts, offsets, both permutations),
    # fp32 token rows [T x H], one add count per (token, 512-column tile), and
    # the mailboxes of its rank-group claims, 2 U + 1024 entries for
    # U = (ceil(T*topk / 256) + E) ceil(H / 512) R
    a256 = lambda b: -(-b // 256) * 256  # noqa: E731
    u1 = (8192 // 256 + 8) * (4096 // 512) * 8
    assert s == (256 + a256(9 * 4) + a256(8 * 4) + a256(9 * 4) + 2 * a256(8192 * 4) + 4096 * 4096 * 4
                 + a256(4096 * 8 * 4) + a256((2 * u1 + 1024) * 4))
    # layer0: header, tile table, a ready count per 256-row unit, the staged rows
    # [T*topk x H] and the mailboxes of its unit schedule, 2 U + 1024 entries for
    # U = (ceil(T*topk / 256) + E)(ceil(F / 512) + R)
    u = (8192 // 256 + 8) * (-(-14336 // 512) + 8)
    m0 = fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, 8, 4096, 4096, 14336, 8, 2)
    assert m0 == 256 + 256 + 256 + 8192 * 4096 * 2 + -(-(2 * u + 1024) * 4 // 256) * 256
    assert fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, 3, 4096, 4096, 14336, 8, 2) == 0
    # the EP x TP split does not change the workspace, and F need not divide by R
    assert fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_RS, 8, 4096, 4096, 14336, 8, 2) == s
    assert fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_AG, 3, 4095, 4096, 14336, 6, 2) > 256
    assert fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_AG, 3, 4096, 4096, 14336, 6, 2) == 0


FAKE = 1 << 20  # never dereferenced: every case below fails validation first


def _err(fx, fn, *args, **kw):
    with pytest.raises(fx.FluxError) as e:
        fn(*args, **kw)
    return e.value.status


def test_host_validation_without_gpu(fx):
    class WS:  # stand-in workspace: only its address and size are looked at
        def __init__(self, n, addr=FAKE):
            self.n, self.addr = n, addr

        def data_ptr(self):
            return self.addr

        def numel(self):
            return self.n

        def element_size(self):
            return 1

    ws = WS(256)
    p = [FAKE] * 8
    S = 0  # explicit stream: the host checks never need CUDA
    assert _err(fx, fx.flux_ag_gemm, 0, 64, 64, 64, fx.FLUX_F16, p, p, p, None, ws, stream=S) == \
        fx.FLUX_ERR_INVALID_ARG
    assert _err(fx, fx.flux_ag_gemm, 17, 68, 68, 64, fx.FLUX_F16, p * 3, p * 3, p * 3, None, ws,
                stream=S) == fx.FLUX_ERR_INVALID_ARG
    assert _err(fx, fx.flux_ag_gemm, 3, 64, 66, 64, fx.FLUX_F16, p, p, p, None, ws, stream=S) == \
        fx.FLUX_ERR_INVALID_ARG
    assert _err(fx, fx.flux_ag_gemm, 2, 64, 64, 64, 7, p, p, p, None, ws, stream=S) == \
        fx.FLUX_ERR_INVALID_ARG
    assert _err(fx, fx.flux_ag_gemm, 2, 64, 64, 64, fx.FLUX_F16, [FAKE, 0], p, p, None, ws,
                stream=S) == fx.FLUX_ERR_INVALID_ARG
    assert _err(fx, fx.flux_ag_gemm, 2, 64, 64, 60, fx.FLUX_F16, p, p, p, None, ws, stream=S) == \
        fx.FLUX_ERR_UNSUPPORTED
    assert _err(fx, fx.flux_ag_gemm, 2, 64, 64, 64, fx.FLUX_F16, [FAKE + 8, FAKE], p, p, None, ws,
                stream=S) == fx.FLUX_ERR_UNSUPPORTED
    assert _err(fx, fx.flux_ag_gemm, 2, 12, 64, 64, fx.FLUX_F16, p, p, p, None, ws, stream=S) == \
        fx.FLUX_ERR_UNSUPPORTED  # 6 rows per shard: no 8-row TMA box fits
    assert _err(fx, fx.flux_gemm, 64, 64, 64, fx.FLUX_F16, FAKE, FAKE, FAKE, WS(255), stream=S) == \
        fx.FLUX_ERR_WORKSPACE
    assert _err(fx, fx.flux_gemm, 64, 64, 64, fx.FLUX_F16, FAKE, FAKE, FAKE, WS(256, FAKE + 16),
                stream=S) == fx.FLUX_ERR_WORKSPACE
    # the least GEMM-RS accepts: header + counters + fp32 rows (no schedule mailboxes)
    need = 256 + 256 + 64 * 64 * 4
    assert need < fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, 2, 64, 64, 64)
    assert _err(fx, fx.flux_gemm_rs, 2, 64, 64, 64, fx.FLUX_F16, p, p, p, WS(need - 1), stream=S) == \
        fx.FLUX_ERR_WORKSPACE
    assert _err(fx, fx.flux_gemm_rs, 2, 63, 64, 64, fx.FLUX_F16, p, p, p, WS(need), stream=S) == \
        fx.FLUX_ERR_INVALID_ARG
    assert _err(fx, fx.flux_gemm_rs, 2, 64, 60, 64, fx.FLUX_F16, p, p, p, WS(need), stream=S) == \
        fx.FLUX_ERR_UNSUPPORTED
    assert _err(fx, fx.flux_moe_route, 8, 0, 2, FAKE, FAKE, FAKE, FAKE, FAKE, stream=S) == \
        fx.FLUX_ERR_INVALID_ARG
    assert _err(fx, fx.flux_moe_route, 8, 2000, 2, FAKE, FAKE, FAKE, FAKE, FAKE, stream=S) == \
        fx.FLUX_ERR_INVALID_ARG
    big = WS(1 << 40)
    assert _err(fx, fx.flux_moe_ag_grouped_gemm, 2, 64, 64, 64, 4, 5, fx.FLUX_F16, p, p, FAKE, p,
                FAKE, FAKE, FAKE, FAKE, None, big, stream=S) == fx.FLUX_ERR_INVALID_ARG  # topk > E
    assert _err(fx, fx.flux_moe_grouped_gemm_rs, 2, 64, 64, 64, 4, 2, fx.FLUX_F16, p, p, FAKE, FAKE,
                FAKE, None, None, p, big, stream=S) == fx.FLUX_ERR_INVALID_ARG  # partial routing
    for tp in (1, 3):  # E = 6 experts over 4 groups; tp = 3 does not divide R = 4
        assert _err(fx, fx.flux_moe_ep_dispatch_gemm, 4, tp, 64, 64, 64, 6, 2, fx.FLUX_F16, p, p,
                    FAKE, p, FAKE, FAKE, FAKE, FAKE, None, big, stream=S) == fx.FLUX_ERR_INVALID_ARG
        assert _err(fx, fx.flux_moe_ep_gemm_combine, 4, tp, 64, 64, 64, 6, 2, fx.FLUX_F16, p, p,
                    FAKE, FAKE, None, None, None, p, big, stream=S) == fx.FLUX_ERR_INVALID_ARG
    assert _err(fx, fx.flux_moe_ep_dispatch_gemm, 4, 2, 64, 64, 60, 4, 2, fx.FLUX_F16, p, p,
                FAKE, p, FAKE, FAKE, FAKE, FAKE, None, big, stream=S) == \
        fx.FLUX_ERR_UNSUPPORTED  # F/tp = 30 columns: rows not 16-byte aligned


def test_valid_call_without_gpu_reports_instead_of_crashing(fx):
    import torch
    if torch.cuda.is_available():
        pytest.skip("this machine has a GPU")
    with pytest.raises(fx.FluxError) as e:
        fx.flux_gemm(64, 64, 64, fx.FLUX_F16, FAKE, FAKE, FAKE, _ws256(), stream=0)
    assert e.value.status in (fx.FLUX_ERR_CUDA, fx.FLUX_ERR_NO_DEVICE)


def _ws256():
    class W:
        def data_ptr(self):
            return FAKE

        def numel(self):
            return 256

        def element_size(self):
            return 1
    return W()


def test_checked_build_exports_the_same_symbols_and_says_so(fx):
    # the checked build (-DFLUX_CHECKS=1) is a drop-in copy of the library
    path = os.path.join(os.path.dirname(fx.LIB_PATH), "libflux_gb300_checked.so")
    assert os.path.exists(path), "build() makes the checked library too"
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} missing from the checked build"
    lib.flux_checks_enabled.restype = ctypes.c_int
    assert lib.flux_checks_enabled() == 1
    regular = ctypes.CDLL(os.path.join(os.path.dirname(fx.LIB_PATH), "libflux_gb300.so"))
    regular.flux_checks_enabled.restype = ctypes.c_int
    assert regular.flux_checks_enabled() == 0
