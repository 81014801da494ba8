"""Throughput of the fused GEMM + tensor-parallel collective hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input,
every rank virtual (R = 8 buffer sets on this GPU):

  dense TP-MLP   AllGather+GEMM  X[4096 x 12288] . W1[12288 x 49152]  (fp16)
                 -> GEMM+ReduceScatter Output1[4096 x 49152] . W2[49152 x 12288]
  decode         GEMM+ReduceScatter act[128 x 28672] . W2[28672 x 8192]  (bf16)
  MoE layer      routing (T=4096, E=8, top-2, Zipf(1.2) bias) -> layer0 AllGather +
                 gather-by-expert grouped GEMM [.. x 4096] . [4096 x 14336] -> layer1
                 grouped GEMM [.. x 14336] . [14336 x 4096] + top-k combine +
                 ReduceScatter (bf16)

Prints ONE JSON line.  ``--impl reference`` times the CPU oracle on this
host's cores instead, on a bounded row sample of the same workload.

The path runs on one GPU: the R ranks are buffer sets in that GPU's memory,
and the dense kernels share operand tiles between the CTAs of a cluster by
TMA multicast, a form kept to single-GPU calls.  With more than one GPU
(``--gpus N`` > 1, or WORLD_SIZE > 1 under torchrun) the arm of this library
prints one line with ``"value": null`` and the reason, and exits without
touching CUDA; the oracle arm (``--impl reference``) runs on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import configs  # noqa: E402

METRIC = "fused AG-GEMM/GEMM-RS TFLOP/s vs fp16 peak; overhead vs plain GEMM (us)"
UNIT = "TFLOP/s"
WORKLOAD = ("hot-path step, R=8 virtual ranks: dense TP-MLP AG-GEMM 4096x12288x49152 -> "
            "GEMM-RS 4096x49152x12288 (fp16); decode GEMM-RS 128x28672x8192 (bf16); "
            "MoE layer T=4096 H=4096 F=14336 E=8: top-2 gate on router scores + routing + "
            "layer0 + layer1 (bf16)")
DTYPE = "f16/bf16 operands, fp32 accumulate"
# the sources that decide what each op's kernel does (device code + the host
# code that fills its parameters); a traffic figure is valid for one hash
KERNEL_SOURCES = {
    "dense": ["flux_kernels.cuh", "flux_ptx.cuh", "flux_dense.cu"],
    "moe": ["flux_kernels.cuh", "flux_ptx.cuh", "flux_moe.cu"],
}


def kernel_hash(op: str = "gemm_rs") -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES["moe" if op.startswith("moe") else "dense"]:
        with open(os.path.join(ROOT, "reducescatter_tcgen05_tmem_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "tc": p["bf16_tflops"], "tc_sus": p["bf16_tflops_sustained"],
                "src": "measured"}
    except Exception:
        return {"hbm": 6800.0, "tc": 1900.0, "tc_sus": 1700.0, "src": "fallback"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 20 ms, timestamped) from before the warm-up to
    the end of the run; summary(t0, t1) reduces the samples taken inside one
    host wall-clock window (the timed region, or one comparison region)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_dir: str = ""):
        import tempfile
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join(out_dir or tempfile.gettempdir(), f"flux_clocks_gpu{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        """End the sampling (the file keeps every sample)."""
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        self.proc = None
        self.done = True

    def summary(self, t0: float, t1: float):
        """Summary of the samples taken between host wall-clock times t0 and t1
        (the sampler may still be running)."""
        import datetime
        if self.proc is None and not getattr(self, "done", False):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        if self.proc is not None:
            self.fh.flush()
        sm, pw, smax, reasons, seen = [], [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    mhz, mx = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                seen += 1
                if not t0 <= ts <= t1:
                    continue
                sm.append(mhz)
                smax = mx
                try:
                    pw.append(float(parts[4]))
                except ValueError:
                    pass
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
               "reasons": sorted(reasons), "samples": len(sm),
               "power_w_median": statistics.median(pw) if pw else None,
               "window_s": round(t1 - t0, 3)}
        if not sm:
            out["note"] = f"no sample inside the timed region ({seen} in the whole run)"
        return out


# ---------------------------------------------------------------- our arm
class Step:
    """Device buffers and the launch sequence of one hot-path step."""

    # the hot-path step (the MoE layer starts from router scores: gate, then
    # routing + layer0, then layer1); the expert-parallel MoE layers on the
    # same workload are extra ops selected with --ops
    STEP_OPS = ["ag_gemm", "gemm_rs", "decode_rs", "moe_gate", "moe_layer0", "moe_layer1"]
    EXTRA_OPS = ["moe_ep_layer0", "moe_ep_layer1"]
    LAUNCHES = {"ag_gemm": 1, "gemm_rs": 1, "decode_rs": 1, "moe_layer0": 2, "moe_layer1": 2,
                "moe_gate": 1, "moe_ep_layer0": 2, "moe_ep_layer1": 2}

    def __init__(self, torch, fx, dev, small=False, ops=None, op_opts=None):
        from workloads.torch_io import to_device
        self.torch, self.fx, self.dev = torch, fx, dev
        # launch options per op (flux_opts_t fields); ops without any use the
        # library's defaults (or what flux_tune_* recorded)
        self.op_opts = dict(op_opts or {})
        self.ops = list(ops) if ops else list(self.STEP_OPS)
        unknown = [o for o in self.ops if o not in self.STEP_OPS + self.EXTRA_OPS]
        if unknown:
            raise SystemExit(f"unknown ops {unknown}")
        want = set(self.ops)
        C = configs.CONFIGS
        ag, rs, dec, moe = C["ag_mlp0"], C["rs_mlp1"], C["rs_decode"], C["moe"]
        if small:  # same structure, reduced sizes with >= 5 waves per op (profiling captures)
            ag = configs.small(ag, N=8 * 768, K=8192)
            rs = configs.small(rs, N=3072, K=8 * 2048)
            dec = configs.small(dec, K=8 * 1792)
            moe = configs.small(moe, T=2048, F=8 * 896)
        self.ag, self.rs, self.dec, self.moe = ag, rs, dec, moe
        T = lambda a, d: to_device(a, d, dev)  # noqa: E731

        def ws(nbytes):
            return torch.zeros(max(nbytes, 256) // 4, dtype=torch.int32, device=dev)
        self.workspaces = []
        t0 = time.time()
        # only the buffers of the selected ops are allocated (a profile of one
        # op then holds that op's memory alone)
        if "ag_gemm" in want:
            xs, w1 = configs.ag_inputs(ag)
            self.X = [T(x, "f16") for x in xs]
            self.W1 = [T(w, "f16") for w in w1]
            del xs, w1
            self.flags = torch.ones(ag.R, dtype=torch.int32, device=dev)
            ag_op = fx.FLUX_OP_AG_GEMM_PUSH if self.op_opts.get("ag_gemm", {}).get("ag_push") \
                else fx.FLUX_OP_AG_GEMM
            self.ws_ag = ws(fx.flux_workspace_size(ag_op, ag.R, ag.M, ag.N, ag.K))
            self.workspaces.append(self.ws_ag)
        if "ag_gemm" in want or "gemm_rs" in want:
            # Output1: written by the AG-GEMM in the chained step, else the
            # GEMM-RS workload's own activations
            if "ag_gemm" in want:
                self.out1 = [torch.empty(ag.M, ag.N // ag.R, dtype=torch.float16, device=dev)
                             for _ in range(ag.R)]
            else:
                a_s, _ = configs.rs_inputs(configs.small(rs, N=8))
                self.out1 = [T(a, "f16") for a in a_s]
                del a_s
        if "gemm_rs" in want:
            _, w2 = configs.rs_inputs(configs.small(rs, M=rs.R * 8))
            self.W2 = [T(w, "f16") for w in w2]
            del w2
            self.out2 = [torch.empty(rs.M // rs.R, rs.N, dtype=torch.float16, device=dev) for _ in range(rs.R)]
            self.ws_rs = ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, rs.R, rs.M, rs.N, rs.K))
            self.workspaces.append(self.ws_rs)
        if "decode_rs" in want:
            da, dw = configs.rs_inputs(dec)
            self.dA = [T(a, "bf16") for a in da]
            self.dW = [T(w, "bf16") for w in dw]
            self.dout = [torch.empty(dec.M // dec.R, dec.N, dtype=torch.bfloat16, device=dev)
                         for _ in range(dec.R)]
            self.ws_dec = ws(fx.flux_workspace_size(fx.FLUX_OP_GEMM_RS, dec.R, dec.M, dec.N, dec.K))
            self.workspaces.append(self.ws_dec)
        moe_ops = {"moe_gate", "moe_layer0", "moe_layer1", "moe_ep_layer0", "moe_ep_layer1"}
        self.has_moe = bool(want & moe_ops)
        if self.has_moe:
            n = moe.T * moe.topk
            tp_layers = want & {"moe_layer0", "moe_layer1"}
            standalone_h = "moe_layer1" in want and "moe_layer0" not in want
            md = configs.moe_inputs(moe, with_h=standalone_h)
            # router scores; the gate writes the routing the layers read
            self.logits = torch.from_numpy(md["logits"]).to(dev)
            self.ids = torch.empty(moe.T, moe.topk, dtype=torch.int32, device=dev)
            self.gw = torch.empty(moe.T, moe.topk, dtype=torch.float32, device=dev)
            self.counts = torch.empty(moe.E, dtype=torch.int32, device=dev)
            self.offsets = torch.empty(moe.E + 1, dtype=torch.int32, device=dev)
            self.s2r = torch.empty(n, dtype=torch.int32, device=dev)
            self.r2s = torch.empty(n, dtype=torch.int32, device=dev)
            self.mflags = torch.ones(moe.R, dtype=torch.int32, device=dev)
            if tp_layers or want & {"moe_ep_layer0"}:
                self.mX = [T(x, "bf16") for x in md["x_shards"]]
            if "moe_layer0" in want:
                self.mW1 = [T(w, "bf16") for w in md["w1_shards"]]
                self.ws_m0 = ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_AG, moe.R, moe.T, moe.H, moe.F,
                                                           moe.E, moe.topk))
                self.workspaces.append(self.ws_m0)
            if tp_layers:
                if standalone_h:  # layer1 alone: the workload's standalone layer1 input
                    self.mH = [T(h, "bf16") for h in md["h_shards"]]
                else:
                    self.mH = [torch.empty(n, moe.F // moe.R, dtype=torch.bfloat16, device=dev)
                               for _ in range(moe.R)]
            if "moe_layer1" in want or "moe_ep_layer1" in want:
                self.mY = [torch.empty(moe.T // moe.R, moe.H, dtype=torch.bfloat16, device=dev)
                           for _ in range(moe.R)]
            if "moe_layer1" in want:
                self.mW2 = [T(w, "bf16") for w in md["w2_shards"]]
                self.ws_m1 = ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_RS, moe.R, moe.T, moe.H, moe.F,
                                                           moe.E, moe.topk))
                self.workspaces.append(self.ws_m1)
            del md
            if want & {"moe_ep_layer0", "moe_ep_layer1"}:
                self.tp = 1
                ed = configs.moe_ep_inputs(moe, self.tp, with_h=False)
                if "moe_ep_layer0" not in want:
                    self.mX = getattr(self, "mX", None) or [T(x, "bf16") for x in ed["x_shards"]]
                self.eW1 = [T(w, "bf16") for w in ed["w1_shards"]]
                self.eW2 = [T(w, "bf16") for w in ed["w2_shards"]]
                del ed
                hbuf = torch.empty(n, moe.F // self.tp, dtype=torch.bfloat16, device=dev)
                self.eH = [hbuf] * moe.R  # one grouped buffer: each rank writes its expert's rows
                self.ws_e0 = ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_AG, moe.R, moe.T, moe.H,
                                                           moe.F, moe.E, moe.topk))
                self.ws_e1 = ws(fx.flux_moe_workspace_size(fx.FLUX_OP_MOE_EP_RS, moe.R, moe.T, moe.H,
                                                           moe.F, moe.E, moe.topk))
                self.workspaces += [self.ws_e0, self.ws_e1]
        self.gen_s = time.time() - t0
        self.flops = {
            "ag_gemm": ag.flops, "gemm_rs": rs.flops, "decode_rs": dec.flops,
            "moe_layer0": moe.flops_per_layer, "moe_layer1": moe.flops_per_layer,
            "moe_ep_layer0": moe.flops_per_layer, "moe_ep_layer1": moe.flops_per_layer,
            "moe_gate": 0.0,
        }
        if self.has_moe:
            # the layers find a routing even when the gate is not timed
            self.run_op("moe_gate")
            if "moe_layer1" in want and "moe_layer0" not in want:
                fx.flux_moe_route(moe.T, moe.E, moe.topk, self.ids, self.counts, self.offsets, self.s2r,
                                  self.r2s)
            if "moe_ep_layer1" in want and "moe_ep_layer0" not in want:
                self.run_op("moe_ep_layer0")
        self.launches_per_step = sum(self.LAUNCHES[o] for o in self.ops)

    def run_op(self, name, extra=None):
        fx, ag, rs, dec, moe = self.fx, self.ag, self.rs, self.dec, self.moe
        o = dict(self.op_opts.get(name, {}))
        o.update(extra or {})
        o = o or None
        if name == "ag_gemm":
            fx.flux_ag_gemm(ag.R, ag.M, ag.N, ag.K, fx.FLUX_F16, self.X, self.W1, self.out1, self.flags,
                            self.ws_ag, opts=o)
        elif name == "gemm_rs":
            fx.flux_gemm_rs(rs.R, rs.M, rs.N, rs.K, fx.FLUX_F16, self.out1, self.W2, self.out2, self.ws_rs,
                            opts=o)
        elif name == "decode_rs":
            fx.flux_gemm_rs(dec.R, dec.M, dec.N, dec.K, fx.FLUX_BF16, self.dA, self.dW, self.dout, self.ws_dec,
                            opts=o)
        elif name == "moe_layer0":
            fx.flux_moe_ag_grouped_gemm(moe.R, moe.T, moe.H, moe.F, moe.E, moe.topk, fx.FLUX_BF16, self.mX,
                                        self.mW1, self.ids, self.mH, self.counts, self.offsets, self.s2r,
                                        self.r2s, self.mflags, self.ws_m0, opts=o)
        elif name == "moe_layer1":
            fx.flux_moe_grouped_gemm_rs(moe.R, moe.T, moe.H, moe.F, moe.E, moe.topk, fx.FLUX_BF16, self.mH,
                                        self.mW2, self.ids, self.gw, self.offsets, self.s2r, self.r2s,
                                        self.mY, self.ws_m1, opts=o)
        elif name == "moe_gate":
            fx.flux_moe_topk_gate(moe.T, moe.E, moe.topk, self.logits, self.ids, self.gw)
        elif name == "moe_ep_layer0":
            fx.flux_moe_ep_dispatch_gemm(moe.R, self.tp, moe.T, moe.H, moe.F, moe.E, moe.topk,
                                         fx.FLUX_BF16, self.mX, self.eW1, self.ids, self.eH,
                                         self.counts, self.offsets, self.s2r, self.r2s, self.mflags,
                                         self.ws_e0, opts=o)
        elif name == "moe_ep_layer1":
            fx.flux_moe_ep_gemm_combine(moe.R, self.tp, moe.T, moe.H, moe.F, moe.E, moe.topk,
                                        fx.FLUX_BF16, self.eH, self.eW2, self.ids, self.gw,
                                        self.offsets, self.s2r, self.r2s, self.mY, self.ws_e1, opts=o)

    def trace(self, out_dir):
        """One traced call of every fused op of the step (flux_opts_t.trace):
        the records go to out_dir/trace_<op>.npy and the summary of each to
        out_dir/trace_summary.json, which is also returned."""
        from reducescatter_tcgen05_tmem_gb300 import trace as ftrace
        torch = self.torch
        os.makedirs(out_dir, exist_ok=True)
        buf = torch.zeros(8 + 8 * 152 * 256, dtype=torch.int64, device=self.dev)
        out = {}
        for name in self.ops:
            if name == "moe_gate":
                continue
            buf.zero_()
            self.run_op(name, {"trace": buf})
            torch.cuda.synchronize()
            self.check_status()
            arr = buf.cpu().numpy()
            np.save(os.path.join(out_dir, f"trace_{name}.npy"), arr)
            out[name] = ftrace.summary(ftrace.records(arr))
        with open(os.path.join(out_dir, "trace_summary.json"), "w") as f:
            json.dump(out, f, indent=1)
        return out

    def tune(self):
        """Record per-problem launch options for this step's ops (flux_tune_*);
        the step's calls pass no options, so they use the recorded ones."""
        fx, ag, rs, dec, moe = self.fx, self.ag, self.rs, self.dec, self.moe
        keep = lambda o: {k: v for k, v in o.items() if v}  # noqa: E731
        chosen = {}
        if "ag_gemm" in self.ops:
            chosen["ag_gemm"] = keep(fx.flux_tune_ag_gemm(ag.R, ag.M, ag.N, ag.K, fx.FLUX_F16, self.X,
                                                          self.W1, self.out1, self.flags, self.ws_ag))
        if "gemm_rs" in self.ops:
            chosen["gemm_rs"] = keep(fx.flux_tune_gemm_rs(rs.R, rs.M, rs.N, rs.K, fx.FLUX_F16, self.out1,
                                                          self.W2, self.out2, self.ws_rs))
        if "decode_rs" in self.ops:
            chosen["decode_rs"] = keep(fx.flux_tune_gemm_rs(dec.R, dec.M, dec.N, dec.K, fx.FLUX_BF16,
                                                            self.dA, self.dW, self.dout, self.ws_dec))
        if "moe_layer0" in self.ops:
            chosen["moe_layer0"] = keep(fx.flux_tune_moe_layer0(
                moe.R, moe.R, moe.T, moe.H, moe.F, moe.E, moe.topk, fx.FLUX_BF16, self.mX, self.mW1,
                self.ids, self.mH, self.counts, self.offsets, self.s2r, self.r2s, self.mflags, self.ws_m0))
        if "moe_layer1" in self.ops:
            chosen["moe_layer1"] = keep(fx.flux_tune_moe_layer1(
                moe.R, moe.R, moe.T, moe.H, moe.F, moe.E, moe.topk, fx.FLUX_BF16, self.mH, self.mW2,
                self.ids, self.gw, self.offsets, self.s2r, self.r2s, self.mY, self.ws_m1))
        return chosen

    def step(self, events=None):
        for name in self.ops:
            if events is not None:
                events[name][0].record()
            self.run_op(name)
            if events is not None:
                events[name][1].record()

    def check_status(self):
        for w in self.workspaces:
            st, rep = self.fx.flux_get_status(w)
            if st != self.fx.FLUX_OK:
                raise RuntimeError(f"device status {st}: {rep}")

    def io_buffers(self):
        """(inputs, outputs) of the selected ops as attribute names: the
        activations that enter the chain from the host every step (weights
        stay resident) and the results that leave it."""
        o = set(self.ops)
        ins, outs = [], []
        if "ag_gemm" in o:
            ins.append("X")
        elif "gemm_rs" in o:
            ins.append("out1")
        if "gemm_rs" in o:
            outs.append("out2")
        elif "ag_gemm" in o:
            outs.append("out1")
        if "decode_rs" in o:
            ins.append("dA")
            outs.append("dout")
        if "moe_gate" in o:
            ins.append("logits")
        if o & {"moe_layer0", "moe_ep_layer0"}:
            ins.append("mX")
        if "moe_layer1" in o:
            outs.append("mY")
            if "moe_layer0" not in o:
                ins.append("mH")
        elif "moe_layer0" in o:
            outs.append("mH")
        if "moe_ep_layer1" in o:
            if "mY" not in outs:
                outs.append("mY")
        elif "moe_ep_layer0" in o:
            outs.append("eH")
        return ins, outs

    def total_flops(self):
        return sum(self.flops[o] for o in self.ops)


def per_expert_gemms(torch, st, op):
    """The MoE layer's GEMMs as plain per-expert cuBLAS calls (no gather, no
    combine, no ReduceScatter): for every rank r and expert e with n_e rows
    routed to it, [n_e x K] . W_r[e] into a slice of a grouped output -- R x E
    matmuls, the unfused baseline of a grouped GEMM.  The routing counts are
    the step's own.  None for other ops."""
    if op not in ("moe_layer0", "moe_layer1"):
        return None
    moe = st.moe
    counts = st.counts[:moe.E].cpu().tolist()
    n = moe.T * moe.topk
    if op == "moe_layer0":
        A = torch.randn(n, moe.H, device=st.dev, dtype=torch.bfloat16)
        Ws = st.mW1  # R x [E x H x F/R]
        outs = [torch.empty(n, moe.F // moe.R, device=st.dev, dtype=torch.bfloat16) for _ in range(moe.R)]
        As = [A] * moe.R
    else:
        As = st.mH   # R x [n x F/R] grouped rows
        Ws = st.mW2  # R x [E x F/R x H]
        outs = [torch.empty(n, moe.H, device=st.dev, dtype=torch.bfloat16) for _ in range(moe.R)]
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + int(c))

    def run():
        for r in range(moe.R):
            for e in range(moe.E):
                lo, hi = offs[e], offs[e + 1]
                if hi > lo:
                    torch.matmul(As[r][lo:hi], Ws[r][e], out=outs[r][lo:hi])
    return run


def compare_plain(torch, fx, st, op, M, N, K, dtype, iters, clocks):
    """The fused op against a plain unsplit GEMM of the same shape, C[M x N] =
    A[M x K] B[K x N] by cuBLAS and by this library's own tcgen05 GEMM (and,
    for the MoE layers, against their per-expert cuBLAS GEMMs), measured in
    the same conditions: one region of `iters` rounds, each round launching
    the fused op, then the plain GEMMs back to back, so that all see the same
    clocks and power limit.  Returns the median CUDA-event time of each
    (after the first round), the region's median SM clock, and time x clock
    (cycles) for each."""
    dev = st.dev
    td = torch.float16 if dtype == "f16" else torch.bfloat16
    A = torch.randn(M, K, device=dev, dtype=td)
    B = torch.randn(K, N, device=dev, dtype=td) * 0.02
    C = torch.empty(M, N, device=dev, dtype=td)
    # the full workspace: the own GEMM runs the dynamic unit schedule, like the fused ops
    ws = torch.zeros(fx.flux_workspace_size(fx.FLUX_OP_GEMM, 1, M, N, K) // 4, dtype=torch.int32,
                     device=dev)
    code = fx.FLUX_F16 if dtype == "f16" else fx.FLUX_BF16
    fns = [("fused", lambda: st.run_op(op)),
           ("cublas", lambda: torch.matmul(A, B, out=C)),
           ("own", lambda: fx.flux_gemm(M, N, K, code, A, B, C, ws))]
    pe = per_expert_gemms(torch, st, op)
    if pe is not None:
        fns.append(("per_expert", pe))
    for _ in range(2):
        for _, fn in fns:
            fn()
    torch.cuda.synchronize()
    n = max(4, iters)
    evs = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)] for k, _ in fns}
    w0 = time.time()
    for i in range(n):
        for k, fn in fns:
            a, b = evs[k][i]
            a.record()
            fn()
            b.record()
    torch.cuda.synchronize()
    w1 = time.time()
    st.check_status()
    st_ws = fx.flux_get_status(ws)
    if st_ws[0] != fx.FLUX_OK:
        raise RuntimeError(f"plain GEMM device status {st_ws}")
    med = {k: statistics.median(a.elapsed_time(b) for a, b in evs[k][1:]) for k, _ in fns}
    del A, B, C, ws, fns, pe
    torch.cuda.empty_cache()
    clk = clocks.summary(w0, w1)
    mhz = clk.get("sm_mhz")
    best = min(med["cublas"], med["own"])
    out = {"fused_us": round(med["fused"] * 1e3, 1), "plain_cublas_us": round(med["cublas"] * 1e3, 1),
           "plain_own_us": round(med["own"] * 1e3, 1),
           "overhead_us": round((med["fused"] - best) * 1e3, 1),
           "overhead_frac": round(med["fused"] / best - 1.0, 4),
           "plain_shape": f"{M}x{N}x{K} {dtype}", "rounds": n,
           "region_s": round(w1 - w0, 3), "sm_mhz": mhz, "reasons": clk.get("reasons")}
    if "per_expert" in med:
        out["plain_per_expert_us"] = round(med["per_expert"] * 1e3, 1)
        out["vs_per_expert_frac"] = round(med["fused"] / med["per_expert"] - 1.0, 4)
    if mhz:
        out["mcycles"] = {k: round(med[k] * 1e-3 * mhz, 3) for k in med}  # ms x MHz = 1e3 x Mcycles / 1e3
    return out


def run_ours(args):
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import reducescatter_tcgen05_tmem_gb300 as fx

    st = Step(torch, fx, dev, small=args.small, ops=args.ops.split(",") if args.ops else None,
              op_opts=json.loads(args.op_opts) if args.op_opts else None)
    tuned = st.tune() if args.tune else None
    clocks = ClockSampler(0, args.clocks_dir)
    clocks.start()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    st.check_status()

    # ------------------------------------------------------------ device-timed region
    per_op = {o: 0.0 for o in st.ops}
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record()
    per_step_events = []
    for _ in range(args.steps):
        ev = {o: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for o in st.ops}
        st.step(ev)
        per_step_events.append(ev)
    t_end.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    time.sleep(0.1)  # the sampler's last lines cover the end of the window
    clk = clocks.summary(wall0, wall1)
    ms_total = t_start.elapsed_time(t_end)
    for ev in per_step_events:
        for o in st.ops:
            per_op[o] += ev[o][0].elapsed_time(ev[o][1])
    st.check_status()
    ms_step = ms_total / args.steps
    flops = st.total_flops()
    value = flops / (ms_step * 1e-3) / 1e12

    # ------------------------------------------------------------ end to end through the public API
    e2e = e2e_measure(torch, st, args, dev)

    # ------------------------------------------------------------ per-unit traces (on request)
    traces = st.trace(args.trace_dir) if args.trace_dir else None

    # ------------------------------------------------------------ overhead vs plain unsplit GEMMs
    overhead = {}
    if not args.no_overhead:
        shapes = {
            "ag_gemm": (st.ag.M, st.ag.N, st.ag.K, "f16"),
            "gemm_rs": (st.rs.M, st.rs.N, st.rs.K, "f16"),
            "decode_rs": (st.dec.M, st.dec.N, st.dec.K, "bf16"),
            "moe_layer0": (st.moe.T * st.moe.topk, st.moe.F, st.moe.H, "bf16"),
            "moe_layer1": (st.moe.T * st.moe.topk, st.moe.H, st.moe.F, "bf16"),
        }
        shapes["moe_ep_layer0"], shapes["moe_ep_layer1"] = shapes["moe_layer0"], shapes["moe_layer1"]
        for o in st.ops:
            if o not in shapes:
                continue
            M, N, K, d = shapes[o]
            overhead[o] = compare_plain(torch, fx, st, o, M, N, K, d, args.steps, clocks)
            overhead[o]["fused_us_in_step"] = round(per_op[o] / args.steps * 1e3, 1)
    clocks.stop()

    pk = peaks()
    breakdown = {o: {"ms": round(per_op[o] / args.steps, 4),
                     "tflops": round(st.flops[o] / (per_op[o] / args.steps * 1e-3) / 1e12, 1)}
                 for o in st.ops}
    breakdown = {o: (v if st.flops[o] else {"ms": v["ms"]}) for o, v in breakdown.items()}
    dom = max(st.ops, key=lambda o: per_op[o])
    dom_ms = per_op[dom] / args.steps
    dom_tf = st.flops[dom] / (dom_ms * 1e-3) / 1e12
    # (the committed DRAM bytes are for the full-size launch: none at reduced sizes)
    traffic = None if args.small else load_traffic(dom)
    # the peak that matches the timed window: the burst figure (a matmul timed
    # alone) for a region under a second, the sustained one (seconds back to
    # back under the power limit) for longer regions
    sustained = ms_total >= 1000.0
    peak = pk["tc_sus"] if sustained else pk["tc"]
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(dom_tf, 1),
                "peak": peak, "unit": "TFLOP/s", "frac": round(dom_tf / peak, 4),
                "peak_kind": (f"bf16 dense, {'sustained' if sustained else 'burst'} ({pk['src']}), "
                              f"chosen for a {ms_total / 1e3:.2f} s timed region "
                              "(sustained from 1 s on); fp16 has the same nominal rate"),
                "traffic": traffic,
                "algorithmic_flops_per_launch": st.flops[dom]}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded normal / Zipf-routed inputs, random-init weights)",
        "config": {"workload": WORKLOAD + (" [reduced sizes]" if args.small else ""),
                   "ops": st.ops,
                   "parallelism": "R=8 virtual TP ranks on one GPU",
                   "l2": "inputs larger than L2 (weights 0.47-1.2 GB per op stream from HBM every step)",
                   "step_tflop": round(flops / 1e12, 3),
                   "dense_kernel_grid": fx.flux_launch_info(fx.FLUX_OP_AG_GEMM, fx.FLUX_F16),
                   "launch_options": ("tuned on this GPU before warm-up (flux_tune_*): "
                                      + json.dumps(tuned, sort_keys=True)) if tuned is not None
                   else ("per op: " + json.dumps(st.op_opts, sort_keys=True)) if st.op_opts
                   else "library defaults"},
        "roofline": roofline,
        "breakdown": breakdown,
        "overhead_vs_plain_gemm": overhead,
        "e2e": e2e,
        "gpu_launches": st.launches_per_step * args.steps,
        **({"trace": traces} if traces is not None else {}),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line), flush=True)


def load_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    ent = d.get(kernel)
    if not ent or ent.get("kernel_hash") != kernel_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


def e2e_measure(torch, st, args, dev):
    """Same metric through the public API with host buffers: every step copies
    its activations and router scores in from pinned host memory and its
    results out to pinned host memory.  Two sets of device input/output
    buffers let the copies of neighbouring steps run on a copy stream while a
    step computes: step i+1's inputs go in and step i-1's results come out
    during step i (the order a serving loop would use); the timed region
    spans the first copy in to the last copy out."""
    in_lists, out_lists = st.io_buffers()
    sets = [{a: getattr(st, a) for a in in_lists + out_lists}, {}]
    for a in in_lists + out_lists:
        v = sets[0][a]
        if isinstance(v, list):
            twin = {}
            sets[1][a] = [twin.setdefault(t.data_ptr(), torch.empty_like(t)) for t in v]
        else:
            sets[1][a] = torch.empty_like(v)

    def _flat(v):
        v = v if isinstance(v, list) else [v]
        seen, out = set(), []
        for t in v:  # a buffer shared by several ranks crosses the link once
            if t.data_ptr() not in seen:
                seen.add(t.data_ptr())
                out.append(t)
        return out

    def dev_in(k):
        return sum((_flat(sets[k][a]) for a in in_lists), [])

    def dev_out(k):
        return sum((_flat(sets[k][a]) for a in out_lists), [])

    host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in dev_in(0)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out(0)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    # as many steps as the device-timed region, so that both run equally long
    # under the power limit
    n = max(3, args.steps)
    comp = torch.cuda.current_stream()
    cp = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def copy_in(i):
        k = i % 2
        with torch.cuda.stream(cp):
            if i >= 2:
                cp.wait_event(comp_done[k])  # step i-2 has read this set's inputs
            for h, d in zip(host_in, dev_in(k)):
                d.copy_(h, non_blocking=True)
            h2d_done[k].record(cp)

    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    cp.wait_event(t0)
    copy_in(0)
    for i in range(n):
        k = i % 2
        if i + 1 < n:
            copy_in(i + 1)
        comp.wait_event(h2d_done[k])
        if i >= 2:
            comp.wait_event(d2h_done[k])  # step i-2's results left this set's outputs
        for a, v in sets[k].items():
            setattr(st, a, v)
        st.step()
        comp_done[k].record(comp)
        with torch.cuda.stream(cp):
            cp.wait_event(comp_done[k])
            for d, h in zip(dev_out(k), host_out):
                h.copy_(d, non_blocking=True)
            d2h_done[k].record(cp)
    for k in range(2):
        comp.wait_event(d2h_done[k])
    t1.record(comp)
    torch.cuda.synchronize()
    for a, v in sets[0].items():
        setattr(st, a, v)
    ms = t0.elapsed_time(t1) / n
    return {"value": round(st.total_flops() / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n,
            "resident": "weights stay resident in HBM; activations, router scores and results cross "
                        "the link every step, double-buffered on a copy stream"}


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)
_SAMPLE_CACHE = {}


def _sample_configs(rows, cols, tokens, fcols):
    """Row/column samples of each op of the step: same K, same rank structure,
    fewer output rows and columns (all drawn by the same seeded generator)."""
    C = configs.CONFIGS
    ag, rs, dec, moe = C["ag_mlp0"], C["rs_mlp1"], C["rs_decode"], C["moe"]
    return (configs.small(ag, M=ag.R * max(rows // ag.R, 1), N=ag.R * cols),
            configs.small(rs, M=rs.R * max(rows // rs.R, 1), N=cols),
            configs.small(dec, N=cols),
            configs.small(moe, T=moe.R * max(tokens // moe.R, 1), F=moe.R * fcols))


def _sample_inputs(key):
    if key not in _SAMPLE_CACHE:
        ag, rs, dec, m = _sample_configs(*key)
        _SAMPLE_CACHE.clear()
        _SAMPLE_CACHE[key] = (configs.ag_inputs(ag), configs.rs_inputs(rs), configs.rs_inputs(dec),
                              configs.moe_inputs(m, with_h=False))
    return _SAMPLE_CACHE[key]


def oracle_sample(rows, cols, tokens, fcols):
    """One bounded CPU-oracle sample of the step (AG-GEMM, GEMM-RS, decode
    GEMM-RS, MoE gate + routing + layer0 + layer1) on a row/column sample of every op.
    Returns (flops, seconds of oracle time; input generation excluded)."""
    import oracle
    ag, rs, dec, m = _sample_configs(rows, cols, tokens, fcols)
    (xs, w1), (As, Bs), (da, dw), md = _sample_inputs((rows, cols, tokens, fcols))
    t = time.time()
    oracle.ag_gemm(xs, w1, ag.dtype)
    oracle.gemm_rs(As, Bs, rs.dtype)
    oracle.gemm_rs(da, dw, dec.dtype)
    ids, gates = oracle.moe_topk_gate(md["logits"], m.topk)
    h, routing = oracle.moe_layer0(md["x_shards"], md["w1_shards"], ids, m.E, m.dtype)
    oracle.moe_layer1(h, md["w2_shards"], ids, gates, m.E, m.dtype, routing_=routing, h_dtype="f64")
    secs = time.time() - t
    flops = ag.flops + rs.flops + dec.flops + 2 * m.flops_per_layer
    return flops, secs


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def _sample_desc(rows, cols, tokens, fcols):
    return (f"float64 numpy oracle on a sample of every op: {rows} token rows x {cols} output "
            f"columns per rank (AG-GEMM, GEMM-RS), 128 x {cols} (decode), {tokens} MoE tokens with "
            f"F/R = {fcols}; full reduction lengths")


def cpu_baseline(args):
    key = (args.cpu_rows, args.cpu_cols, args.cpu_tokens, args.cpu_fcols)
    flops, secs = oracle_sample(*key)
    return {"value": round(flops / secs / 1e12, 5), "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": _sample_desc(*key) + f" ({flops / 1e9:.1f} GFLOP in {secs:.1f} s)"}


def run_reference(args):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    key = (args.ref_rows, args.ref_cols, args.ref_tokens, args.ref_fcols)
    for _ in range(args.warmup):
        oracle_sample(*key)
    tot_f, tot_s = 0.0, 0.0
    t0 = time.time()
    for _ in range(args.steps):
        f, s = oracle_sample(*key)
        tot_f += f
        tot_s += s
    wall = time.time() - t0
    value = tot_f / tot_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "sample": _sample_desc(*key)},
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": _cores(), "kind": "oracle",
                         "sample": "each step: " + _sample_desc(*key)},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # defaults: a timed region of about one second (sustained clocks and power)
    ap.add_argument("--steps", type=int, default=120)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--small", action="store_true", help="reduced sizes (profiling captures)")
    ap.add_argument("--ops", default="", help="comma list of ops to run (default: the whole step)")
    ap.add_argument("--no-overhead", action="store_true")
    ap.add_argument("--tune", action="store_true",
                    help="record per-problem launch options (flux_tune_*) before the warm-up")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op-opts", default="",
                    help='launch options per op as JSON, e.g. \'{"gemm_rs": {"rs_tile": 2}}\'')
    ap.add_argument("--trace-dir", default="",
                    help="after the timed region, trace one call of each fused op into this directory")
    ap.add_argument("--clocks-dir", default="",
                    help="where the raw nvidia-smi samples are written (default: the temp dir)")
    ap.add_argument("--cpu-rows", type=int, default=512)
    ap.add_argument("--cpu-cols", type=int, default=8192)
    ap.add_argument("--cpu-tokens", type=int, default=2048)
    ap.add_argument("--cpu-fcols", type=int, default=1024)
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--ref-cols", type=int, default=512)
    ap.add_argument("--ref-tokens", type=int, default=128)
    ap.add_argument("--ref-fcols", type=int, default=128)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    ws_, rank, _ = dist_env()
    n = max(args.gpus, ws_)
    if n > 1:
        # single-GPU path: nothing of this library is launched on more than one
        # GPU (and CUDA is not initialised here)
        if rank == 0:
            print(json.dumps(single_gpu_only_line(args, n)), flush=True)
        return
    run_ours(args)


def single_gpu_only_line(args, n):
    """The line printed for a multi-GPU request: the path has no multi-GPU form."""
    return {"metric": METRIC, "value": None, "unit": UNIT, "n_gpus": n, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE, "data": "synthetic",
            "config": {"workload": WORKLOAD, "parallelism": "R=8 virtual TP ranks on one GPU"},
            "unavailable": ("single-GPU path: the R tensor-parallel ranks are buffer sets on one GPU, "
                            "and its dense kernels share operand tiles inside a cluster by TMA "
                            "multicast, which is kept to 1-GPU calls; no multi-GPU form is built")}


if __name__ == "__main__":
    main()
