#!/usr/bin/env python
"""Benchmark of the routed top-k MoE experts forward on GB300.

One step = one pass of the whole path over one synthetic batch: router top-k
(moe_route), then the experts forward (dispatch, grouped gate/up GEMM with
SwiGLU, grouped down GEMM with the weighted combine, bf16 output).  Weights
and inputs are resident in HBM when the timed region starts (``value``);
``e2e`` repeats the measurement through host buffers with the copies inside
the timed region.

Default workload: the DeepSeek-V3-shaped layer in prefill (T=8192, H=7168,
I=2048, E=256, k=8, Zipf(1.1) expert skew), bf16, the largest of the
single-GPU workloads.  ``--workload`` selects another one.

Under torchrun each rank runs an independent replica on its own GPU (the
path has no exchange step); ``value`` is the tokens of all ranks divided by
the slowest rank's time.

``--impl reference`` times the CPU oracle (the plain eager expert loop) on
the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE experts fwd tokens/s, TFLOP/s or HBM GB/s as fraction of 1-GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# name -> (shape name, T, weight format, scale format)
WORKLOADS = {
    "qwen-prefill": ("qwen", 4096, "bf16", None),
    "tiny": ("tiny", 64, "bf16", None),
    "qwen-decode-1": ("qwen", 1, "bf16", None),
    "qwen-decode-8": ("qwen", 8, "bf16", None),
    "qwen-decode-32": ("qwen", 32, "bf16", None),
    "qwen-decode-128": ("qwen", 128, "bf16", None),
    "dsv3-prefill": ("dsv3", 8192, "bf16", None),
    "dsv3-fp8-64-f32": ("dsv3_fp8", 64, "fp8", "f32"),
    "dsv3-fp8-64-ue8m0": ("dsv3_fp8", 64, "fp8", "ue8m0"),
    "dsv3-fp8-16384-f32": ("dsv3_fp8", 16384, "fp8", "f32"),
    "dsv3-fp8-16384-ue8m0": ("dsv3_fp8", 16384, "fp8", "ue8m0"),
    # profiling-sized layers (32 experts), used for ncu captures
    "dsv3e32-fp8-2048-f32": ("dsv3_e32", 2048, "fp8", "f32"),
    "dsv3e32-fp8-8-f32": ("dsv3_e32", 8, "fp8", "f32"),
    "dsv3e32-fp8-2048-ue8m0": ("dsv3_e32", 2048, "fp8", "ue8m0"),
    "dsv3e32-fp4-2048": ("dsv3_e32", 2048, "fp4", "ue8m0"),
    "dsv3e32-prefill": ("dsv3_e32", 2048, "bf16", None),
    # FP4 (e2m1, 1x32 UE8M0 blocks) experts: GEMVs up to 64 routed rows,
    # block-scaled tensor-core GEMMs above
    "qwen-fp4-decode-1": ("qwen", 1, "fp4", "ue8m0"),
    "qwen-fp4-decode-16": ("qwen", 16, "fp4", "ue8m0"),
    "dsv3-fp4-1": ("dsv3", 1, "fp4", "ue8m0"),
    "dsv3-fp4-8": ("dsv3", 8, "fp4", "ue8m0"),
    "qwen-fp4-prefill": ("qwen", 4096, "fp4", "ue8m0"),
    "dsv3-fp4-prefill": ("dsv3", 8192, "fp4", "ue8m0"),
}
DESCRIPTIONS = {
    "qwen": "Qwen1.5-MoE-A2.7B-shaped MoE layer",
    "tiny": "tiny MoE FFN",
    "dsv3": "DeepSeek-V3-shaped MoE layer, Zipf(1.1) expert skew",
    "dsv3_fp8": "DeepSeek-V3-shaped MoE layer, Zipf(1.1) skew, e4m3 128x128 block-scaled weights",
    "dsv3_e32": "DeepSeek-V3-width MoE layer with 32 experts (profiling size)",
}
L2_BYTES = 129 * 2 ** 20
BYTES_PER_WEIGHT = {"bf16": 2.0, "fp8": 1.0, "fp4": 0.5}
WDTYPE = {"bf16": 0, "fp8": 1, "fp4": 2}
DTYPE_NAME = {"bf16": "bf16", "fp8": "fp8-e4m3", "fp4": "fp4-e2m1"}


def describe(name):
    sname, _, wfmt, sfmt = WORKLOADS[name]
    d = DESCRIPTIONS[sname]
    if wfmt == "fp4":
        return d + ", packed e2m1 weights with 1x32 UE8M0 scales"
    if wfmt == "fp8" and "e4m3" not in d:
        return d + f", e4m3 weights with 128x128 {sfmt} scales"
    return d


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.isfile(p):
        try:
            d = json.load(open(p))
            return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML every few ms."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x10: "sync_boost"}

    def __init__(self, cuda_index: int):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.ok = False
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            busid = self._bus_id(cuda_index)
            if busid is None or nv.nvmlDeviceGetHandleByPciBusId_v2(busid, ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(h)) != 0:
                    return
            self.nv, self.h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except Exception:
            self.ok = False

    @staticmethod
    def _bus_id(i):
        try:
            import torch
            p = torch.cuda.get_device_properties(i)
            return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
        except Exception:
            return None

    def _loop(self):
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if self._reason_fn(self.h, ctypes.byref(r)) == 0:
                for bit, name in self.REASONS.items():
                    if r.value & bit:
                        self.reasons.add(name)
            time.sleep(0.005)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._loop, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples), "source": "nvml"}


# ------------------------------------------------------------------ ranks
def max_over_ranks(x: float, device) -> float:
    """Largest value of x over all ranks (identity without a process group).
    Each rank runs an independent replica; the job's time is the slowest."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank processed its own batch of
    tokens_per_step in each of the steps; the job took the slowest rank's
    max_ms milliseconds."""
    return world * tokens_per_step * steps / (max_ms / 1e3)


# ------------------------------------------------------------------ workload
def build_workload(name, device):
    import torch
    import mixture_experts_routed_top_gb300 as moe
    from workloads import make_inputs, shape_for
    sname, T, wfmt, sfmt = WORKLOADS[name]
    shape = shape_for(sname, T)
    d = make_inputs(shape, seed=0, device=device)
    w = {"shape": shape, "wfmt": wfmt, "sfmt": sfmt, "logits": d["logits"],
         "hidden": d["hidden"], "w_gate_up": d["w_gate_up"], "w_down": d["w_down"]}
    if wfmt == "fp8":
        w["q_gate_up"], w["s_gate_up"] = moe.quantize_fp8_blocks(d["w_gate_up"], sfmt)
        w["q_down"], w["s_down"] = moe.quantize_fp8_blocks(d["w_down"], sfmt)
        torch.cuda.synchronize()
    elif wfmt == "fp4":
        w["q_gate_up"], w["s_gate_up"] = moe.quantize_fp4_blocks(d["w_gate_up"])
        w["q_down"], w["s_down"] = moe.quantize_fp4_blocks(d["w_down"])
        torch.cuda.synchronize()
    return w


def weights_of(w):
    if w["wfmt"] in ("fp8", "fp4"):
        return dict(w_gate_up=w["q_gate_up"], w_down=w["q_down"], scale_gate_up=w["s_gate_up"],
                    scale_down=w["s_down"], scale_fmt=w["sfmt"])
    return dict(w_gate_up=w["w_gate_up"], w_down=w["w_down"])


def tensor_ratio(w):
    """Nominal tensor rate of the path's MMAs over the bf16 rate."""
    return 2.0 if w["wfmt"] in ("fp8", "fp4") else 1.0


def dominant_roof(w, dominant, flops, wbytes, peaks):
    """Algorithmic work of the dominant GEMM stage and the roof that binds it.

    The gate/up GEMM does 2/3 of the step's flops and weight bytes, the down
    GEMM 1/3.  Its algorithmic bytes are its weights, its activations in and
    its result out once (gate/up: the routed rows of X in, h out; down: h
    in, the fp32 [T, H] accumulator out).  The roofline time is the larger
    of flops / tensor peak and bytes / HBM bandwidth; the kernel is reported
    against that roof.  The tensor peak is the measured sustained bf16 rate
    (x2 for the FP8-rate MMAs): every timed region is a loop of back-to-back
    steps, so the kernel runs as the sustained measurement did, against the
    power cap.  Returns (flops, bytes, weight bytes, tensor peak in TFLOP/s,
    hbm_bound)."""
    s = w["shape"]
    share = (2.0 / 3.0) if dominant == "gemm1" else (1.0 / 3.0)
    kern_flops = flops * share
    kern_wbytes = wbytes * share
    rows = s.T * s.k
    act_b = 2.0 if w["wfmt"] == "bf16" else 1.0
    if dominant == "gemm1":
        kern_bytes = kern_wbytes + rows * s.H * act_b + rows * s.I * act_b
    else:
        kern_bytes = kern_wbytes + rows * s.I * act_b + s.T * s.H * 4.0
    # e4m3 x e4m3 and e4m3 x e2m1 (kind::mxf8f6f4) run at the FP8 rate
    pk = peaks["bf16_tflops_sustained"] * tensor_ratio(w)
    hbm_bound = kern_bytes / (peaks["hbm_gbs"] * 1e9) >= kern_flops / (pk * 1e12)
    return kern_flops, kern_bytes, kern_wbytes, pk, hbm_bound


def roof_entry(w, hbm_bound, kern_flops, kern_bytes, d_avg_s, pk, peaks):
    """The dominant kernel against the roof that binds it: its algorithmic
    bytes or flops per launch over its average launch time.  Tensor-bound
    entries are against `pk` (the sustained rate, from dominant_roof) and
    carry the fraction of the burst rate beside it."""
    if hbm_bound:
        achieved = kern_bytes / d_avg_s / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
    achieved = kern_flops / d_avg_s / 1e12
    pk_burst = peaks["bf16_tflops"] * tensor_ratio(w)
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk,
            "unit": "TFLOP/s", "frac": round(achieved / pk, 4),
            "frac_of_burst": round(achieved / pk_burst, 4), "peak_burst": pk_burst}


def algorithmic(w, counts):
    """Algorithmic flops and bytes of one step (routed rows only; weight bytes
    of the experts that received rows; hidden in, logits in, output out)."""
    s = w["shape"]
    rows = s.T * s.k
    flops = 6.0 * s.H * s.I * rows
    bpw = BYTES_PER_WEIGHT[w["wfmt"]]
    touched = int((counts > 0).sum())
    scale_b = 0
    if w["wfmt"] == "fp8":
        per = 4 if w["sfmt"] == "f32" else 1
        scale_b = (2 * s.I // 128) * (s.H // 128) * per + (s.H // 128) * (s.I // 128) * per
    elif w["wfmt"] == "fp4":   # one UE8M0 byte per 32 weights
        scale_b = 2 * s.I * (s.H // 32) + s.H * (s.I // 32)
    wbytes = touched * (3.0 * s.H * s.I * bpw + scale_b)
    io = s.T * s.H * 2 * 2 + s.T * s.E * 4
    return flops, wbytes, io, touched


def traffic_for(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.isfile(p):
        return None
    try:
        d = json.load(open(p))
        ent = d.get(kernel_key)
        if not ent:
            return None
        src = os.path.join(ROOT, ent["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return ent["bytes_per_launch"] if h == ent["source_sha"] else None
    except Exception:
        return None


# ------------------------------------------------------------------ CPU oracle
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = [i for i in threadpool_info() if i.get("user_api") == "blas"]
        if info:
            return int(info[0]["num_threads"])
    except Exception:
        pass
    env = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(env) if env else os.cpu_count()


class OracleSample:
    """The CPU oracle (route + eager expert loop in float64) on the first n
    tokens of the workload, with only the experts those tokens select copied
    to the host (at most max_experts of them)."""

    def __init__(self, w, n, max_experts=None):
        import numpy as np
        import torch
        import oracle as O
        self.O, self.w = O, w
        s = w["shape"]
        if max_experts is None:   # about 8 GB of host copies at float32
            max_experts = max(8, int(8e9 // (3 * s.H * s.I * 4)))
        logits = w["logits"].float().cpu().numpy()
        idx_all, _ = O.route(logits, s.k)
        toks, ex = [], set()
        for t in range(s.T):
            new = ex | set(int(e) for e in idx_all[t])
            if toks and (len(new) > max_experts or len(toks) >= n):
                break
            toks.append(t)
            ex = new
        toks, ex = np.array(toks), sorted(ex)
        et = torch.tensor(ex, device=w["hidden"].device)
        if w["wfmt"] in ("fp8", "fp4"):
            self.parts = [w["q_gate_up"].index_select(0, et).cpu().numpy(),
                          w["s_gate_up"].index_select(0, et).cpu().numpy(),
                          w["q_down"].index_select(0, et).cpu().numpy(),
                          w["s_down"].index_select(0, et).cpu().numpy()]
        else:
            self.parts = [w["w_gate_up"].index_select(0, et).float().cpu().numpy(),
                          w["w_down"].index_select(0, et).float().cpu().numpy()]
        self.hid = w["hidden"][torch.from_numpy(toks).to(w["hidden"].device)].float().cpu().numpy()
        self.logits = logits[toks]
        self.remap = np.full(s.E, -1, np.int64)
        self.remap[np.array(ex)] = np.arange(len(ex))
        self.n = len(toks)
        self.k = s.k

    def run(self) -> float:
        O = self.O
        t0 = time.perf_counter()
        idx, wt = O.route(self.logits, self.k)
        lidx = self.remap[idx].astype("int32")
        act = self.w.get("act", "silu")
        if self.w["wfmt"] == "fp8":
            O.forward_fp8(self.hid, lidx, wt, *self.parts, self.w["sfmt"], act=act)
        elif self.w["wfmt"] == "fp4":
            O.forward_fp4(self.hid, lidx, wt, *self.parts, act=act)
        else:
            O.forward(self.hid, lidx, wt, *self.parts, act=act)
        return time.perf_counter() - t0


def calibrated_oracle_sample(w, budget_s):
    """Grow the token sample until one oracle run takes about budget_s."""
    s = w["shape"]
    n = 16
    smp = OracleSample(w, n)
    dt = smp.run()
    while dt < budget_s / 2 and smp.n < s.T:
        want = int(min(s.T, max(2 * smp.n, smp.n * budget_s / max(dt, 1e-3) * 0.8)))
        nxt = OracleSample(w, want)
        if nxt.n <= smp.n:
            break
        smp = nxt
        dt = smp.run()
    return smp, dt


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import mixture_experts_routed_top_gb300 as moe
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    moe.lib(build_if_missing=True)
    moe.set_swap_rows({"auto": -1, "rows": 0, "swap": 1 << 20}[args.bf16_gemm])
    moe.set_block_scaled_mma(args.ue8m0_kernel == "block-scaled")
    if args.tile_group is not None:
        moe.set_tile_group(args.tile_group)
    if args.down_phases is not None:
        moe.set_down_phases(args.down_phases)
    if args.pair_gemm is not None:
        moe.set_pair_gemm(args.pair_gemm)
    if args.down_l2 is not None:
        moe.set_down_l2_hints(args.down_l2)
    if args.fp4_gemv_rows is not None:
        moe.set_fp4_gemv_rows(args.fp4_gemv_rows)
    if args.decode_kernels is not None:
        moe.set_decode_single(args.decode_kernels == 1)
    if args.decode_rows is not None:
        moe.set_decode_rows(args.decode_rows)
    w = build_workload(args.workload, dev)
    w["act"] = args.activation
    s = w["shape"]
    W = weights_of(w)
    ws = moe.Workspace(dev)
    out = torch.empty(s.T, s.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(logits, hidden, dst=None):
        idx, wt = moe.route(logits, s.k)
        moe.experts_forward(hidden, idx, wt, out=out if dst is None else dst, workspace=ws,
                            activation=args.activation, **W)
        return idx

    # routing statistics of the workload (outside any timed region)
    idx = step(w["logits"], w["hidden"])
    torch.cuda.synchronize()
    moe.workspace_status(ws)
    counts = torch.bincount(idx.flatten().long(), minlength=s.E).cpu().numpy()
    flops, wbytes, io_bytes, touched = algorithmic(w, counts)
    ws_bytes = moe.workspace_size(s.T, s.H, s.I, s.E, s.k, WDTYPE[w["wfmt"]])
    working_set = wbytes + io_bytes
    flush = working_set < 2 * L2_BYTES
    flush_buf = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev) if flush else None

    for _ in range(args.warmup):
        if flush:
            flush_buf.zero_()
        step(w["logits"], w["hidden"])
    torch.cuda.synchronize()

    graph = graph_prof = None
    if args.graph:
        # One step (router + forward, every kernel of the library) captured
        # as a CUDA graph for the timed region, and a second capture of the
        # same step with per-stage CUDA events for the per-kernel durations:
        # the event nodes add several microseconds per stage, so they stay
        # out of the timed steps.
        n_cap = moe.launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(w["logits"], w["hidden"])
        per_step_launches = moe.launch_count() - n_cap
        moe.profile_begin()
        graph_prof = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_prof):
            step(w["logits"], w["hidden"])
        for _ in range(args.warmup):
            graph.replay()
            graph_prof.replay()
        torch.cuda.synchronize()

    def timed_steps(profiled):
        """K steps with the L2 flush between them; per-step CUDA events on the
        launching stream. With profiled=True the stage events are on too and
        their sums are returned."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        acc = {}
        if profiled and graph is None:
            moe.profile_begin()
        for i in range(args.steps):
            if flush:
                flush_buf.zero_()
            starts[i].record(stream)
            if graph is not None:
                (graph_prof if profiled else graph).replay()
            else:
                step(w["logits"], w["hidden"])
            ends[i].record(stream)
            if profiled and graph is not None:
                torch.cuda.synchronize()
                for k_, (ms_, n_) in moe.profile_read().items():
                    a_ = acc.get(k_, (0.0, 0))
                    acc[k_] = (a_[0] + ms_, a_[1] + n_)
        torch.cuda.synchronize()
        if profiled:
            ended = moe.profile_end()
            if graph is None:
                acc = ended
        return [a.elapsed_time(b) for a, b in zip(starts, ends)], acc

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    n0 = moe.launch_count()
    with ClockSampler(dev.index) as clk:
        step_ms, _ = timed_steps(profiled=False)
    launches = (per_step_launches * args.steps) if graph is not None else moe.launch_count() - n0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(sum(step_ms), dev)
    # per-stage kernel durations: the same K steps again, with stage events
    _, stages = timed_steps(profiled=True)
    moe.workspace_status(ws)

    # ---------------------------------------------------------- end to end
    h_host = w["hidden"].cpu().pin_memory()
    l_host = w["logits"].cpu().pin_memory()
    o_host = torch.empty(s.T, s.H, dtype=torch.bfloat16).pin_memory()
    h_dev = torch.empty_like(w["hidden"])
    l_dev = torch.empty_like(w["logits"])

    def e2e_step():
        h_dev.copy_(h_host, non_blocking=True)
        l_dev.copy_(l_host, non_blocking=True)
        step(l_dev, h_dev)
        o_host.copy_(out, non_blocking=True)

    for _ in range(max(2, args.warmup // 2)):
        e2e_step()
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e_start.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), dev)
    e2e_outs = {"serial": o_host.clone()}

    # The same, overlapped as a serving loop would run it: step i+1's inputs
    # go host -> device on one copy stream and step i-1's output device ->
    # host on another while step i computes; inputs and outputs are double
    # buffered and events order every reuse.
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    hb = [torch.empty_like(w["hidden"]) for _ in range(2)]
    lb = [torch.empty_like(w["logits"]) for _ in range(2)]
    ob = [torch.empty_like(out) for _ in range(2)]
    oh = [torch.empty(s.T, s.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def overlapped(nsteps, t_start=None):
        if t_start is not None:
            s_in.wait_event(t_start)
            s_out.wait_event(t_start)
        for i in range(nsteps):
            b = i & 1
            if i >= 2:
                s_in.wait_event(ev_done[b])       # step i-2 has read buffer b
            with torch.cuda.stream(s_in):
                hb[b].copy_(h_host, non_blocking=True)
                lb[b].copy_(l_host, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])      # step i-2's output has left ob[b]
            step(lb[b], hb[b], dst=ob[b])
            ev_done[b].record(stream)
            s_out.wait_event(ev_done[b])
            with torch.cuda.stream(s_out):
                oh[b].copy_(ob[b], non_blocking=True)
                ev_out[b].record(s_out)
        stream.wait_event(ev_out[(nsteps - 1) & 1])
        if nsteps >= 2:
            stream.wait_event(ev_out[nsteps & 1])

    # The same once more as one CUDA graph per step: the pinned host ->
    # device copies, the router and forward calls and the device -> host copy
    # of the output, captured once and replayed every step (how a decode loop
    # is usually run).
    e2e_graph_ms = None
    if args.graph:
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_step()
        for _ in range(max(2, args.warmup // 2)):
            g_e2e.replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gs.record(stream)
        for _ in range(args.steps):
            g_e2e.replay()
        ge.record(stream)
        torch.cuda.synchronize()
        e2e_graph_ms = max_over_ranks(gs.elapsed_time(ge), dev)
        e2e_outs["graph"] = o_host.clone()

    overlapped(max(2, args.warmup // 2))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    o_start, o_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    o_start.record(stream)
    overlapped(args.steps, o_start)
    o_end.record(stream)
    torch.cuda.synchronize()
    e2e_ov_ms = max_over_ranks(o_start.elapsed_time(o_end), dev)
    # every end-to-end loop's output agrees with the device-resident run: the
    # fp32 combine's order may move a bf16 rounding by one unit at the
    # largest outputs (~2 % of rms), far below what a torn or stale buffer
    # gives
    ref_out = out.float().cpu()
    rms = ref_out.pow(2).mean().sqrt().item() or 1.0
    e2e_outs["overlapped"] = oh[(args.steps - 1) & 1]
    for name, got in e2e_outs.items():
        dev_max = (got.float() - ref_out).abs().max().item()
        if dev_max > 5e-2 * rms:
            raise RuntimeError(f"{name} end-to-end output differs from the device-resident run "
                               f"(max |diff| {dev_max:.3g}, rms {rms:.3g})")

    # ---------------------------------------------------------- report
    peaks, peak_src = load_peaks()
    ms_per_step = total_ms / args.steps
    tok_s = job_throughput(s.T, args.steps, world, total_ms)
    g1_ms, g1_n = stages["gemm1"]
    g2_ms, g2_n = stages["gemm2"]
    dominant = "gemm1" if g1_ms >= g2_ms else "gemm2"
    d_ms, d_n = stages[dominant]
    d_avg_s = d_ms / max(d_n, 1) / 1e3
    kern_flops, kern_bytes, kern_wbytes, pk, hbm_bound = dominant_roof(w, dominant, flops, wbytes,
                                                                      peaks)
    roof = roof_entry(w, hbm_bound, kern_flops, kern_bytes, d_avg_s, pk, peaks)
    peak_kind = ("hbm_gbs, STREAM-style copy" if hbm_bound else
                 "bf16 sustained: the kernel runs inside a loop of back-to-back steps"
                 if w["wfmt"] == "bf16" else
                 "bf16 sustained x2 nominal fp8/bf16 ratio: the kernel runs inside a loop of "
                 "back-to-back steps")
    mx_path = (w["wfmt"] == "fp8" and w["sfmt"] == "ue8m0" and moe.get_block_scaled_mma()) or \
              (w["wfmt"] == "fp4" and s.T * s.k > moe.get_fp4_gemv_rows())
    # the same kernel against the other roof (both matter near the ridge)
    if w["wfmt"] == "fp4" and not mx_path:
        # the FP4 GEMVs run their multiply-adds on CUDA cores: fp32 FMA peak
        # = SMs x 128 lanes x 2 flops x the largest SM clock seen
        props = torch.cuda.get_device_properties(dev)
        clk_max = (clk.summary() or {}).get("sm_max_mhz") or 2070
        pk_a = props.multi_processor_count * 128 * 2 * float(clk_max) * 1e6 / 1e12
        a_a = kern_flops / d_avg_s / 1e12
        roof_other = {"bound": "alu", "achieved": round(a_a, 2), "peak": round(pk_a, 1),
                      "unit": "TFLOP/s", "frac": round(a_a / pk_a, 4),
                      "peak_source": "fp32 FMA on CUDA cores, SM count x 128 x 2 x max SM clock"}
    elif hbm_bound:
        a_t = kern_flops / d_avg_s / 1e12
        roof_other = {"bound": "tensor", "achieved": round(a_t, 1), "peak": pk,
                      "unit": "TFLOP/s", "frac": round(a_t / pk, 4)}
    else:
        a_b = kern_bytes / d_avg_s / 1e9
        roof_other = {"bound": "hbm", "achieved": round(a_b, 1), "peak": peaks["hbm_gbs"],
                      "unit": "GB/s", "frac": round(a_b / peaks["hbm_gbs"], 4)}
    kernel_key = f"{dominant}:{args.workload}"
    roof.update({"traffic": traffic_for(kernel_key), "kernel": dominant,
                 "peak_source": f"{peak_src} ({peak_kind})",
                 "algorithmic_per_launch": {"flops": kern_flops, "bytes": kern_bytes,
                                            "weight_bytes": kern_wbytes},
                 "avg_launch_ms": round(d_avg_s * 1e3, 4)})
    e2e_tok_s = job_throughput(s.T, args.steps, world, e2e_ms)
    e2e_ov_tok_s = job_throughput(s.T, args.steps, world, e2e_ov_ms)
    e2e_loops = {"serial": e2e_tok_s, "overlapped": e2e_ov_tok_s}
    if e2e_graph_ms is not None:
        e2e_loops["graph"] = job_throughput(s.T, args.steps, world, e2e_graph_ms)
    best_loop = max(e2e_loops, key=e2e_loops.get)
    line = {
        "metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_NAME[w["wfmt"]], "data": "synthetic",
        "config": {"workload": args.workload, "description": describe(args.workload),
                   "T": s.T, "H": s.H, "I": s.I, "E": s.E, "k": s.k,
                   "scale_fmt": w["sfmt"], "parallelism": f"replicas x{world}",
                   "l2": ("flushed before every timed step (512 MB write)" if flush else
                          f"inputs larger than L2 ({working_set / 1e9:.2f} GB touched per step)"),
                   "experts_touched": touched, "max_expert_rows": int(counts.max()),
                   "bf16_gemm": args.bf16_gemm, "tile_group": moe.get_tile_group(),
                   "decode_kernels": 1 if moe.get_decode_single() else 2,
                   "decode_rows": moe.get_decode_rows(),
                   "down_phases": moe.get_down_phases(),
                   "pair_gemm": moe.get_pair_gemm(),
                   "down_l2_hints": moe.get_down_l2_hints(),
                   "activation": args.activation,
                   "scaled_kernels": ("block-scaled tensor-core MMA (kind::mxf8f6f4, UE8M0)"
                                      if mx_path else
                                      "CUDA-core GEMVs" if w["wfmt"] == "fp4" else
                                      "software promotion of per-K-block partial sums"
                                      if w["wfmt"] == "fp8" else None),
                   "timed_steps": "CUDA graph replays of one captured step" if args.graph
                                  else "steps launched from Python",
                   "stage_timing": ("per-stage CUDA events in a second capture of the same "
                                    "step, replayed K times after the timed region")
                                   if args.graph else
                                   "per-stage CUDA events in K more steps after the timed region",
                   "workspace_bytes": ws_bytes},
        "tflops": round(flops / (ms_per_step / 1e3) / 1e12, 2),
        "weight_gbs": round(wbytes / (ms_per_step / 1e3) / 1e9, 1),
        "roofline": roof,
        "roofline_other": roof_other,
        "step_ms_percentiles": {q: round(float(np.percentile(step_ms, p_)), 5)
                                for q, p_ in (("p10", 10), ("p50", 50), ("p90", 90))},
        "stages_ms_per_step": {k: round(v[0] / max(v[1], 1), 5) for k, v in stages.items()},
        "e2e": {"value": round(e2e_loops[best_loop], 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h_host.numel() * 2 + l_host.numel() * 4),
                "d2h_bytes_per_step": int(o_host.numel() * 2),
                "loop": best_loop,
                **{f"{k}_value": round(v, 1) for k, v in e2e_loops.items()},
                "how": "pinned host buffers, copied in and the output copied out every step; "
                       "serial: router + experts_forward called from Python, one stream, copy "
                       "in, compute, copy out; overlapped: the same calls, inputs in and output "
                       "out on two copy streams, double buffered, beside the neighbouring "
                       "steps' compute; graph: copies and calls captured once as a CUDA graph "
                       "and replayed every step; value = the fastest loop"},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    return line, w


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="dsv3-prefill", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch every timed step from Python instead of replaying a CUDA graph")
    ap.add_argument("--bf16-gemm", default="auto", choices=["auto", "rows", "swap"],
                    help="orientation of the bf16 grouped GEMMs (library default: auto)")
    ap.add_argument("--ue8m0-kernel", default="block-scaled", choices=["block-scaled", "promotion"],
                    help="FP8 experts with UE8M0 scales: tensor-core block scaling (library "
                         "default) or the software promotion kernel")
    ap.add_argument("--down-phases", type=int, default=None,
                    help="output-column slices of the down GEMMs (library default: automatic)")
    ap.add_argument("--fp4-gemv-rows", type=int, default=None,
                    help="FP4 routed rows at or below which the GEMVs run (library default 64)")
    ap.add_argument("--decode-kernels", type=int, default=None, choices=[1, 2],
                    help="small bf16 decode batches as one cooperative kernel or two kernels "
                         "(library default)")
    ap.add_argument("--decode-rows", type=int, default=None,
                    help="routed rows at or below which the bf16 decode GEMVs run "
                         "(library default 16)")
    ap.add_argument("--down-l2", type=int, default=None, choices=[0, 1, 2, 3],
                    help="down GEMM L2 policies: bit 0 accumulator evict_last, bit 1 weights "
                         "evict_first (library default)")
    ap.add_argument("--pair-gemm", type=int, default=None, choices=[0, 1, 2, 3],
                    help="bf16 grouped GEMMs on CTA pairs: bit 0 gate/up, bit 1 down "
                         "(library default)")
    ap.add_argument("--tile-group", type=int, default=None,
                    help="m-tiles per tile group of the token-row gate/up GEMM (library default)")
    ap.add_argument("--activation", default="silu", choices=["silu", "gelu", "relu"],
                    help="gate activation: SwiGLU (default), GeGLU or ReGLU experts")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args)

    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line, w = run_ours(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp, _ = calibrated_oracle_sample(w, budget_s=8.0)
        # the same sample repeated until about 10 s of CPU work are timed
        reps, dt = 0, 0.0
        while reps == 0 or dt < 10.0:
            dt += smp.run()
            reps += 1
        line["cpu_baseline"] = {"value": round(reps * smp.n / dt, 2), "unit": "tokens/s",
                                "cores": blas_threads(), "kind": "oracle",
                                "sample": f"first {smp.n} tokens of the workload (route + "
                                          f"float64 eager expert loop), run {reps} times, "
                                          f"{dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_reference(args):
    """Reference arm: the CPU oracle as it stands, timed on the host cores;
    each step is the same bounded sample of the workload."""
    import torch
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    if WORKLOADS[args.workload][2] in ("fp8", "fp4") and dev.type != "cuda":
        print(json.dumps({"impl": "reference",
                          "unavailable": "the quantised workload builds its weights with the GPU quantiser"}))
        return 0
    w = build_workload(args.workload, dev)
    w["act"] = args.activation
    s = w["shape"]
    smp, _ = calibrated_oracle_sample(w, budget_s=2.0)
    for _ in range(args.warmup):
        smp.run()
    total = sum(smp.run() for _ in range(args.steps))
    value = smp.n * args.steps / total
    line = {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": args.workload,
                       "description": describe(args.workload),
                       "T": s.T, "H": s.H, "I": s.I, "E": s.E, "k": s.k,
                       "scale_fmt": w["sfmt"], "activation": args.activation},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                             "cores": blas_threads(), "kind": "oracle",
                             "sample": f"each step: first {smp.n} tokens of the workload "
                                       f"(route + float64 eager expert loop)"},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
