#!/usr/bin/env python
"""Benchmark of the MXFP4 MoE layer (route -> permute -> gate_up -> down -> combine).

One step = one pass of the whole layer over one batch of the workload's
tokens, every kernel from libmoe.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload skewed_prefill8192]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

The headline workload (default: the 8192-token skewed prefill, the largest
single-GPU configuration) is timed over exactly K steps.  On rank 0 the line
also carries `per_config`: every other full-size workload (the 64-token
decode step, the 288-token MTP verify step, the 1536-token prefill chunk and
the calibrated skewed prefill) and the headline workload again, each timed
over a region of at least --config-seconds with its own clock record and
binding roofline.

Under torchrun every rank runs its own replica of the layer on its own batch
(the layer is data parallel over tokens; no collective on the data path);
the value is all ranks' tokens divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 MoE layer tokens/s; % of HBM roofline (decode) / tensor peak (prefill)"
DEFAULT_WORKLOAD = "skewed_prefill8192"
# the full-size workloads; each is timed in per_config
PER_CONFIG = ("decode64", "mtp_verify288", "prefill1536", "skewed_prefill8192",
              "skewed_prefill8192_cal")
# bf16 layer: the tile height each full-size workload runs with (decode path
# with 8-row tiles while most experts see a few rows; prefill path above)
BENCH_TILE_M = {"decode64": 8, "mtp_verify288": 8, "prefill1536": 64,
                "skewed_prefill8192": 128, "skewed_prefill8192_cal": 128}
CLOCK_PERIOD_MS = 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=0,
                   help="timed steps (default 0: as many as fill about 2 s, at least 50; the "
                        "reference arm takes 50)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--tile-m", type=int, default=0,
                   help="rows per expert tile (default: bf16 by BENCH_TILE_M, else 8; mxfp4 by "
                        "the mean rows per expert: 32 below 16, 64 below 64, else 128)")
    p.add_argument("--E", type=int, default=0,
                   help="routed experts override (smaller cases for profiler captures)")
    p.add_argument("--path", default="auto", choices=["auto", "decode", "prefill", "prefill_fp8x2"])
    p.add_argument("--replicas", type=int, default=2,
                   help="weight/input replicas rotated per step (keeps L2 cold)")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--act", default="bf16", choices=["bf16", "mxfp4"],
                   help="activations: bf16 (the layer as specified) or MXFP4-quantised "
                        "(moe_ffn_mxfp4act, block-scaled MXFP4 x MXFP4 GEMMs)")
    p.add_argument("--config-seconds", type=float, default=2.0,
                   help="minimum timed region of each per_config entry")
    p.add_argument("--no-per-config", action="store_true")
    return p.parse_args()


# ------------------------------------------------------------------ env

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            return json.load(f)
    except Exception:
        return None


def _find_number(d, keys):
    if isinstance(d, dict):
        for k, v in d.items():
            if k in keys and isinstance(v, (int, float)):
                return float(v)
        for v in d.values():
            r = _find_number(v, keys)
            if r is not None:
                return r
    return None


def hbm_peak():
    mp = measured_peaks()
    if mp is not None:
        v = _find_number(mp, ("hbm_gbs", "hbm_GBps", "copy_gbs"))
        if v:
            return v, "measured (MEASURED_PEAKS.json hbm_gbs)"
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


def tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s (burst: kernels are timed alone)."""
    mp = measured_peaks()
    if mp is not None:
        v = _find_number(mp, ("bf16_tflops",))
        if v:
            return v, "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, earlier GB300 measurement)"


# nominal dense FP4 / BF16 tensor rate on GB300 (13.5 / 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0


def roofline_entry(kernel, bytes_, flops, seconds, traffic, traffic_src, fp4=False):
    """The binding roofline of one kernel: whichever of HBM bytes and tensor
    flops needs more time at peak.  fp4: the contraction runs on MXFP4
    operands, so its peak is the bf16 peak times the nominal FP4/BF16 ratio."""
    hbm, hbm_src = hbm_peak()
    ten, ten_src = tensor_peak()
    if fp4:
        ten, ten_src = ten * FP4_OVER_BF16, f"derived: {ten_src} x {FP4_OVER_BF16:g} (nominal FP4/BF16)"
    t_hbm = bytes_ / (hbm * 1e9)
    t_ten = flops / (ten * 1e12)
    hbm_ach = bytes_ / seconds / 1e9
    ten_ach = flops / seconds / 1e12
    if t_ten > t_hbm:
        bound, ach, peak, unit, src = "tensor", ten_ach, ten, "TFLOP/s", ten_src
    else:
        bound, ach, peak, unit, src = "hbm", hbm_ach, hbm, "GB/s", hbm_src
    return {"kernel": kernel, "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
            "frac": ach / peak, "traffic": traffic,
            "algorithmic_bytes_per_launch": int(bytes_), "flops_per_launch": int(flops),
            "launch_us": seconds * 1e6, "peak_source": src, "traffic_source": traffic_src,
            "hbm_frac": hbm_ach / hbm, "tensor_frac": ten_ach / ten}


def traffic_from_profiles(kernel: str, workload: str, src_file: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (sha256 recorded in the summary)."""
    sha = hashlib.sha256(open(src_file, "rb").read()).hexdigest()[:16]
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        txt = open(path).read()
        for m in re.finditer(r"traffic_bytes_per_launch kernel=(\S+) workload=(\S+) "
                             r"src_sha256=(\S+) bytes=(\d+)", txt):
            if m.group(1) == kernel and m.group(2) == workload and m.group(3) == sha:
                return int(m.group(4)), os.path.relpath(path, ROOT)
    return None, None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every CLOCK_PERIOD_MS."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.out = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(CLOCK_PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(2 * CLOCK_PERIOD_MS / 1e3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        bus = torch.cuda.get_device_properties(device_index).pci_bus_id
        if bus:
            return str(bus)
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[device_index]
    return str(device_index)


# ------------------------------------------------------- algorithmic work

def layer_work(w, ids_host, act="bf16"):
    """Algorithmic HBM bytes and flops of one step, from the actual routing
    (the per-unit figures of the layer: each touched expert's packed weights
    once, x read, h written once and read once, out written, logits read).
      gate_up step: W13 of the touched experts + x read + h write
      down step:    W2 of the touched experts + h read + out write
    Intermediate buffers an implementation adds (f16 copies of rows, the
    per-pair fp32 outputs before the combine) are not algorithmic and are not
    counted.  act="mxfp4": h moves as MXFP4 (codes + scales)."""
    import numpy as np
    from mxfp4_mixture_experts_softmax_gb300 import synth
    touched = int(np.unique(ids_host).size)
    H, I, T, P = w.H, w.I, w.T, w.pairs
    w13_b = 2 * I * (H // 2 + H // 32)
    w2_b = H * (I // 2 + I // 32)
    hb = I // 2 + I // 32 if act == "mxfp4" else 2 * I   # bytes of one h row
    gate_up = touched * w13_b + T * H * 2 + P * hb
    down = touched * w2_b + P * hb + T * H * 2
    layer = touched * synth.weight_bytes_per_expert(w) + T * H * 4 + 2 * P * hb + T * w.E * 4
    flops = 2 * P * (2 * I * H + H * I)
    return dict(touched=touched, gate_up_bytes=gate_up, down_bytes=down, layer_bytes=layer,
                flops=flops, gate_up_flops=2 * P * 2 * I * H)


def workload_config(w, act: str, ws: int) -> dict:
    """The keys that name the workload, shared by both arms' config."""
    return {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "K": w.K,
            "shared_expert": w.with_shared, "Et": w.Et, "Kt": w.Kt,
            "activations": "mxfp4 (OCP MX quantisation of x and h)" if act == "mxfp4" else "bf16",
            "parallelism": f"replicas x{ws} (weak scaling, tokens per GPU fixed)"}


def launches_per_step(w, path_name: str) -> int:
    """Kernel launches of one step: route + permute (one fused launch up to
    MOE_ROUTE_PERMUTE_FUSED_MAX_T tokens; else the routing kernel and the
    permutation, one launch or, for large batches, the four-launch multi-block
    sort), then per path:
      decode   x -> f16 rows, gate_up, h -> f16 rows | down, combine
      prefill  gather of x into tile order as f16 rows, gate_up, h -> f16
               rows | position weights, down, blocked combine
      prefill_fp8x2  gather of x into tile order as two E4M3 terms, gate_up |
               position weights, down, blocked combine
      mxfp4act quantise x, gather, gate_up | position weights, down, blocked
               combine"""
    from mxfp4_mixture_experts_softmax_gb300 import libmoe
    P = w.T * w.Kt
    if w.T <= libmoe.MOE_ROUTE_PERMUTE_FUSED_MAX_T:
        rp = 1
    else:
        nb = min(P // max(w.Et, 1), 160)
        rp = 1 + (4 if (nb >= 8 and P >= 8192) else 1)
    return rp + {"decode": 3 + 2, "prefill": 3 + 3, "prefill_fp8x2": 2 + 3, "mxfp4act": 3 + 3}[path_name]


# ------------------------------------------------------------ ranks

def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings (the slowest rank sets the time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def weak_scaling_value(tokens_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """All ranks' tokens divided by the slowest rank's time (tokens/s)."""
    return tokens_per_rank_step * steps * world / (max_ms / 1e3)


# ------------------------------------------------------------ our arm

def default_tile_m(w, act: str) -> int:
    if act == "bf16":
        return BENCH_TILE_M.get(w.name, 8)
    rows = w.T * w.Kt / w.Et
    return 32 if rows < 16 else 64 if rows < 64 else 128


class Layer:
    """One workload resident on the device: R weight / input replicas rotated
    per step (the touched weights of one step are far larger than L2, and a
    step never finds the previous step's weights there), the routing and
    workspace buffers, and the step itself."""

    def __init__(self, w, act: str, tm: int, path_arg: str, replicas: int, dev):
        import numpy as np
        import torch
        from mxfp4_mixture_experts_softmax_gb300 import libmoe, synth
        self.w, self.act, self.tm, self.dev = w, act, tm, dev
        self.mx = act == "mxfp4"
        self.path = {"auto": libmoe.MOE_PATH_AUTO, "decode": libmoe.MOE_PATH_DECODE,
                     "prefill": libmoe.MOE_PATH_PREFILL,
                     "prefill_fp8x2": libmoe.MOE_PATH_PREFILL_FP8X2}[path_arg]
        resolved = (libmoe.moe_ffn_auto_path_shape(w.T, w.H, w.I, w.Et, w.Kt, tm)
                    if self.path == libmoe.MOE_PATH_AUTO else self.path)
        if self.mx:
            self.path_name = "mxfp4act"
        else:
            self.path_name = {libmoe.MOE_PATH_DECODE: "decode", libmoe.MOE_PATH_PREFILL: "prefill",
                              libmoe.MOE_PATH_PREFILL_FP8X2: "prefill_fp8x2"}[resolved]
        self.host = synth.make_inputs(w)

        def up(a):
            t = torch.from_numpy(np.ascontiguousarray(a))
            if a.dtype == np.uint16:
                t = t.view(torch.int16).view(torch.bfloat16)
            return t.to(dev)

        self.R = max(1, replicas)
        self.weights = [{k: up(self.host[k]) for k in ("w13", "s13", "w2", "s2")}]
        for _ in range(self.R - 1):
            self.weights.append({k: v.clone() for k, v in self.weights[0].items()})
        self.logits = [up(self.host["logits"]) for _ in range(self.R)]
        self.xs = [up(self.host["x"]) for _ in range(self.R)]
        self.bufs = libmoe.alloc_layer(w.T, w.E, w.K, w.with_shared, w.H, w.I, w.Et, tm, dev)
        if self.mx:  # the MXFP4-activation workspace replaces the bf16 one
            self.bufs["workspace"] = libmoe.alloc_workspace_mxfp4act(w.T, w.H, w.I, w.Et, w.Kt,
                                                                     tm, dev)
        self.stream = torch.cuda.current_stream(dev)

    def step(self, i, ev=None, kern_ev=None):
        """One pass of the layer.  ev: events between all calls (breakdown);
        kern_ev: four events the library records around the gate_up and the
        down GEMM kernel launches themselves (moe_set_gemm_events)."""
        from mxfp4_mixture_experts_softmax_gb300 import libmoe
        w, b, r = self.w, self.bufs, i % self.R
        W = self.weights[r]
        if ev is not None:
            ev[0].record(self.stream)
        # routing + permutation: one launch up to MOE_ROUTE_PERMUTE_FUSED_MAX_T tokens
        _, tw, perm = libmoe.moe_route_permute(self.logits[r], w.K, self.tm, w.with_shared,
                                               w.renormalize, b["topk_ids"], b["topk_w"],
                                               b["perm"])
        if ev is not None:
            ev[1].record(self.stream)
        if kern_ev is not None:
            libmoe.moe_set_gemm_events(kern_ev[0], kern_ev[1])
        if self.mx:
            libmoe.moe_ffn_mxfp4act_gate_up(self.xs[r], W["w13"], W["s13"], perm, b["workspace"])
        else:
            libmoe.moe_ffn_gate_up(self.xs[r], W["w13"], W["s13"], perm, b["workspace"],
                                   self.path)
        if ev is not None:
            ev[2].record(self.stream)
        if kern_ev is not None:
            libmoe.moe_set_gemm_events(kern_ev[2], kern_ev[3])
        if self.mx:  # down GEMM and the combine into out
            libmoe.moe_ffn_mxfp4act_down(W["w2"], W["s2"], tw, perm, b["workspace"], w.T, b["out"])
        else:
            libmoe.moe_ffn_down_combine(W["w2"], W["s2"], tw, perm, b["workspace"], w.T, b["out"],
                                        self.path)
        if ev is not None:
            ev[3].record(self.stream)
        if kern_ev is not None:
            libmoe.moe_set_gemm_events(None, None)

    def timed(self, steps: int, gpu_index: int, ws: int = 1, kernel_events: bool = True):
        """Exactly `steps` steps between two events, barrier + synchronize on
        both sides, clocks sampled during the region; returns the region's
        milliseconds, the mean GEMM kernel times (kernel_events: the library
        records a pair of events around each of the two GEMM kernel launches
        of every step, on the launching stream; otherwise nothing is recorded
        inside the region) and the clock record."""
        import torch
        dev = self.dev
        kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        if kernel_events:
            for kv in kevs:  # created before the region (torch creates events on first record)
                for e in kv:
                    e.record(self.stream)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(gpu_id_for(gpu_index))
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t0.record(self.stream)
        for i in range(steps):
            self.step(i, kern_ev=kevs[i] if kernel_events else None)
        t1.record(self.stream)
        torch.cuda.synchronize(dev)
        if ws > 1:
            torch.distributed.barrier()
        clocks = sampler.stop()
        gemm = {}
        if kernel_events:
            gemm = {"gate_up_gemm": statistics.mean(k[0].elapsed_time(k[1]) for k in kevs),
                    "down_gemm": statistics.mean(k[2].elapsed_time(k[3]) for k in kevs)}
        return t0.elapsed_time(t1), gemm, clocks

    def breakdown(self, n: int = 10) -> dict:
        """Per-call times (events between every call; after the timed region)."""
        import torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for i in range(n):
            self.step(i, ev=evs[i])
        torch.cuda.synchronize(self.dev)
        names = ["route_permute", "gate_up", "down"]
        return {nm: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n))
                for j, nm in enumerate(names)}

    def e2e(self, steps: int, warmup: int) -> float:
        """The layer through the public API with host buffers, run as a serving
        loop runs it: every step copies its logits + x from pinned host memory
        (upload stream), runs the layer (the layer's stream) and copies its
        output back to pinned host memory (download stream).  Inputs and
        outputs are double-buffered, so step i + 1's upload and step i - 1's
        download overlap step i's kernels; events order each buffer's reuse.
        Weight replicas rotate as in the device-timed loop.  Returns the
        milliseconds from the first upload to the last download."""
        import torch
        from mxfp4_mixture_experts_softmax_gb300 import libmoe
        w, dev = self.w, self.dev
        ref_out = self.bufs["out"].cpu()  # the device-timed loop's output
        pin_logits = torch.from_numpy(self.host["logits"]).pin_memory()
        pin_x = torch.from_numpy(self.host["x"]).view(torch.int16).view(torch.bfloat16).pin_memory()
        pin_out = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        d_logits = [self.logits[0], torch.empty_like(self.logits[0])]
        d_x = [self.xs[0], torch.empty_like(self.xs[0])]
        bufs = [self.bufs, dict(self.bufs, out=torch.empty_like(self.bufs["out"]))]
        up_s, down_s, cs = torch.cuda.Stream(dev), torch.cuda.Stream(dev), self.stream

        def ev():
            return torch.cuda.Event()
        uploaded = [ev(), ev()]   # inputs j on the device
        consumed = [ev(), ev()]   # layer j done with its inputs and its output written
        downloaded = [ev(), ev()] # output j read back
        used = [False, False]

        def one(i):
            j, W, b = i % 2, self.weights[i % self.R], bufs[i % 2]
            with torch.cuda.stream(up_s):
                if used[j]:
                    up_s.wait_event(consumed[j])
                d_logits[j].copy_(pin_logits, non_blocking=True)
                d_x[j].copy_(pin_x, non_blocking=True)
                uploaded[j].record(up_s)
            cs.wait_event(uploaded[j])
            if used[j]:
                cs.wait_event(downloaded[j])
            if self.mx:
                _, tw, perm = libmoe.moe_route_permute(d_logits[j], w.K, self.tm, w.with_shared,
                                                       w.renormalize, b["topk_ids"], b["topk_w"],
                                                       b["perm"])
                libmoe.moe_ffn_mxfp4act(d_x[j], W["w13"], W["s13"], W["w2"], W["s2"], tw, perm,
                                        b["out"], b["workspace"])
            else:
                libmoe.moe_layer(d_logits[j], d_x[j], W["w13"], W["s13"], W["w2"], W["s2"], w.K,
                                 w.with_shared, w.renormalize, tile_m=self.tm, path=self.path,
                                 bufs=b)
            consumed[j].record(cs)
            with torch.cuda.stream(down_s):
                down_s.wait_event(consumed[j])
                pin_out[j].copy_(b["out"], non_blocking=True)
                downloaded[j].record(down_s)
            used[j] = True

        for i in range(max(3, warmup)):
            one(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        up_s.wait_event(e0)
        for i in range(steps):
            one(i)
        cs.wait_stream(down_s)
        e1.record(cs)
        torch.cuda.synchronize(dev)
        # the deterministic layer gives the device-timed loop's bytes: a
        # buffer reused too early would show here
        last = pin_out[(steps - 1) % 2]
        if not torch.equal(last.view(torch.int16), ref_out.view(torch.int16)):
            raise RuntimeError(f"end-to-end output differs from the device-timed output on {w.name}")
        return e0.elapsed_time(e1)

    def e2e_serial(self, steps: int, warmup: int) -> float:
        """The same through the public API with every copy serialised with the
        layer on one stream (upload, layer, download, then the next step);
        returns ms."""
        import torch
        from mxfp4_mixture_experts_softmax_gb300 import libmoe
        w, b = self.w, self.bufs
        pin_logits = torch.from_numpy(self.host["logits"]).pin_memory()
        pin_x = torch.from_numpy(self.host["x"]).view(torch.int16).view(torch.bfloat16).pin_memory()
        pin_out = torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory()

        def one(i):
            W = self.weights[i % self.R]
            self.logits[0].copy_(pin_logits, non_blocking=True)
            self.xs[0].copy_(pin_x, non_blocking=True)
            if self.mx:
                _, tw, perm = libmoe.moe_route_permute(self.logits[0], w.K, self.tm, w.with_shared,
                                                       w.renormalize, b["topk_ids"], b["topk_w"],
                                                       b["perm"])
                libmoe.moe_ffn_mxfp4act(self.xs[0], W["w13"], W["s13"], W["w2"], W["s2"], tw, perm,
                                        b["out"], b["workspace"])
            else:
                libmoe.moe_layer(self.logits[0], self.xs[0], W["w13"], W["s13"], W["w2"], W["s2"],
                                 w.K, w.with_shared, w.renormalize, tile_m=self.tm, path=self.path,
                                 bufs=b)
            pin_out.copy_(b["out"], non_blocking=True)

        for i in range(max(3, warmup)):
            one(i)
        torch.cuda.synchronize(self.dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for i in range(steps):
            one(i)
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1)

    def check_output(self):
        import numpy as np
        if not np.isfinite(self.bufs["out"].float().cpu().numpy()).all():
            raise RuntimeError(f"non-finite layer output on {self.w.name}")

    def rooflines(self, work, gemm_ms: dict, total_ms: float, steps: int):
        """The gate_up and down GEMM kernels (each timed alone by the events
        the library records around its launch), the gate_up and down +
        combine steps (every launch of each call) and the whole step, each
        against its binding roofline.  The work is the algorithmic work of the
        step either way: the steps' other launches (f16 row copies, the
        combine) add no algorithmic bytes."""
        src = {"prefill": "ffn_prefill.cu", "decode": "ffn_decode.cu",
               "prefill_fp8x2": "ffn_fp8x2.cu", "mxfp4act": "ffn_mxfp4act.cu"}[self.path_name]
        traffic, traffic_src = traffic_from_profiles(
            f"{self.path_name}_gate_up", self.w.name,
            os.path.join(ROOT, "mxfp4_mixture_experts_softmax_gb300", "csrc", src))
        down_flops = work["flops"] - work["gate_up_flops"]
        gu = roofline_entry(f"{self.path_name}_gate_up_gemm", work["gate_up_bytes"],
                            work["gate_up_flops"], gemm_ms["gate_up_gemm"] / 1e3, traffic,
                            traffic_src, fp4=self.mx)
        dn = roofline_entry(f"{self.path_name}_down_gemm", work["down_bytes"], down_flops,
                            gemm_ms["down_gemm"] / 1e3, None, None, fp4=self.mx)
        steps_rl = {
            "gate_up_step": roofline_entry(f"{self.path_name}_gate_up_step", work["gate_up_bytes"],
                                           work["gate_up_flops"], gemm_ms["gate_up"] / 1e3, None,
                                           None, fp4=self.mx),
            "down_combine_step": roofline_entry(f"{self.path_name}_down_combine_step",
                                                work["down_bytes"], down_flops,
                                                gemm_ms["down"] / 1e3, None, None, fp4=self.mx)}
        layer = roofline_entry("layer", work["layer_bytes"], work["flops"], total_ms / steps / 1e3,
                               None, None, fp4=self.mx)
        return gu, dn, layer, steps_rl

    def free(self):
        import torch
        self.weights = self.logits = self.xs = self.bufs = self.host = None
        torch.cuda.empty_cache()


def config_entry(lay, total_ms, steps, gemm, clocks, per, work):
    gu, dn, layer, steps_rl = lay.rooflines(work, gemm, total_ms, steps)
    return {"workload": lay.w.name, "T": lay.w.T, "tile_m": lay.tm, "path": lay.path_name,
            "steps": steps, "timed_s": total_ms / 1e3, "ms_per_step": total_ms / steps,
            "tokens_per_s": lay.w.T * steps / (total_ms / 1e3),
            "experts_touched": work["touched"], "roofline": layer,
            "gate_up_gemm": gu, "down_gemm": dn, **steps_rl,
            "kernels_us": {n: v * 1e3 for n, v in {**per, **gemm}.items()}, "clocks": clocks}


def measure_per_config(args, local, dev, skip=()):
    """Every full-size workload, each timed over at least --config-seconds."""
    import torch
    from mxfp4_mixture_experts_softmax_gb300 import synth
    out = {}
    for name in PER_CONFIG:
        if name in skip:
            continue
        w = synth.WORKLOADS[name]
        lay = Layer(w, args.act, default_tile_m(w, args.act), "auto", args.replicas, dev)
        for i in range(3):
            lay.step(i)
        torch.cuda.synchronize(dev)
        ms, _, _ = lay.timed(5, local, kernel_events=False)
        steps = int(min(20000, max(20, -(-args.config_seconds * 1e3 // (ms / 5)))))
        ids_host = lay.bufs["topk_ids"].cpu().numpy()
        work = layer_work(w, ids_host, args.act)
        # throughput over a region with nothing recorded inside it; the GEMM
        # kernel times over a second, shorter region with the kernel events
        total_ms, _, clocks = lay.timed(steps, local, kernel_events=False)
        _, gemm, _ = lay.timed(max(20, steps // 4), local, kernel_events=True)
        per = lay.breakdown()
        gemm.update(per)
        lay.check_output()
        out[name] = config_entry(lay, total_ms, steps, gemm, clocks, per, work)
        lay.free()
        del lay
    return out


def run_ours(args, ws, rank, local):
    import torch
    from mxfp4_mixture_experts_softmax_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo",
                                device_id=dev if torch.cuda.is_available() else None)
    w = synth.WORKLOADS[args.workload]
    tm = args.tile_m or default_tile_m(w, args.act)  # the full workload's tile height
    if args.E:  # fewer routed experts (profiler captures): same tile height
        w = synth.scaled(w, E=args.E, name=f"{w.name}_E{args.E}")
    lay = Layer(w, args.act, tm, args.path, args.replicas, dev)

    for i in range(args.warmup):
        lay.step(i)
    torch.cuda.synchronize(dev)
    ids_host = lay.bufs["topk_ids"].cpu().numpy()
    work = layer_work(w, ids_host, args.act)

    K = args.steps
    if K <= 0:  # enough steps for a region of about 2 s (the clock sampler's record)
        ms, _, _ = lay.timed(5, local, ws, kernel_events=False)
        K = int(min(20000, max(50, -(-2000.0 // (ms / 5)))))
        if ws > 1:
            K = int(max_over_ranks([K], dev)[0])
    total_ms, gemm, clocks = lay.timed(K, local, ws)
    per = lay.breakdown(min(K, 10))
    gemm.update(per)  # the gate_up and down steps (every launch of each call)
    lay.check_output()
    e2e_ms = lay.e2e(K, args.warmup)
    e2e_serial_ms = lay.e2e_serial(K, args.warmup)
    if ws > 1:
        total_ms, e2e_ms, e2e_serial_ms = max_over_ranks([total_ms, e2e_ms, e2e_serial_ms], dev)

    result = None
    if rank == 0:
        gu, dn, layer, steps_rl = lay.rooflines(work, gemm, total_ms, K)
        result = {
            "metric": METRIC,
            "value": weak_scaling_value(w.T, K, ws, total_ms),
            "unit": "tokens/s",
            "n_gpus": ws,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": total_ms / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            # MMA operand type (f16 rows scaled per row, fp32 accumulation)
            "dtype": "e2m1" if lay.mx else "f16",
            "data": "synthetic (seeded; random MXFP4 weights, N(0,1) activations and logits)",
            "config": {
                **workload_config(w, args.act, ws), "tile_m": tm, "path": lay.path_name,
                "experts_touched": work["touched"],
                "l2": f"inputs larger than L2: {work['layer_bytes'] / 1e9:.2f} GB touched per "
                      f"step, {lay.R} weight replicas rotated per step",
            },
            "roofline": gu,
            "roofline_down": dn,
            "roofline_steps": steps_rl,
            "layer_roofline": layer,
            "kernels_us": {n: v * 1e3 for n, v in {**per, **gemm}.items()},
            # copies on their own streams overlapping the neighbouring steps'
            # kernels (a serving loop); `serial`: each step's copies and layer
            # in order on one stream
            "e2e": {"value": w.T * K * ws / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": int(lay.host["logits"].nbytes + lay.host["x"].nbytes),
                    "d2h_bytes_per_step": int(w.T * w.H * 2),
                    "ms_per_step": e2e_ms / K,
                    "overlap": "uploads and downloads on their own streams, double-buffered",
                    "serial": {"value": w.T * K * ws / (e2e_serial_ms / 1e3),
                               "ms_per_step": e2e_serial_ms / K}},
            "gpu_launches": launches_per_step(w, lay.path_name) * K,
            "clocks": clocks,
        }
    host = lay.host
    lay.free()
    del lay
    if rank == 0 and ws == 1 and not args.no_per_config and not args.E:
        result["per_config"] = measure_per_config(args, local, dev)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, host, None, args.cpu_seconds, args.act)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return result


# ---------------------------------------------------------- the oracle

def _oracle_sample(w, host, ids, wt, n_tokens, threads, offset=0, act="bf16"):
    import numpy as np
    import oracle
    toks = ((np.arange(n_tokens) + offset) % w.T).astype(np.int32)
    fn = oracle.ffn_mxfp4act if act == "mxfp4" else oracle.ffn
    t0 = time.perf_counter()
    fn(host["x"], host["w13"], host["s13"], host["w2"], host["s2"], ids, wt, tokens=toks,
       n_threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w, host, ids_unused, target_s, act="bf16"):
    """The CPU oracle as it stands, timed on this host's cores on a bounded
    sample of the same workload (whole tokens: routing plus all Kt experts)."""
    import oracle
    from mxfp4_mixture_experts_softmax_gb300 import synth
    threads = synth.cpu_threads()
    t0 = time.perf_counter()
    ids, wt = oracle.route(host["logits"], w.K, w.with_shared, w.renormalize)
    route_s = time.perf_counter() - t0
    n = threads
    dt = _oracle_sample(w, host, ids, wt, n, threads, act=act)
    total_tok, total_s = n, dt
    while total_s < target_s and total_tok < 32 * w.T:
        n2 = max(threads, int(n * (target_s - total_s) / max(dt, 1e-3)) // threads * threads)
        n2 = min(n2, 32 * w.T - total_tok)
        dt = _oracle_sample(w, host, ids, wt, n2, threads, offset=total_tok, act=act)
        total_tok += n2
        total_s += dt
    per_tok_route = route_s / w.T
    value = total_tok / (total_s + per_tok_route * total_tok)
    return {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{total_tok} tokens of {w.name} (all {w.Kt} experts each, plus routing), "
                      f"{total_s:.1f} s on {threads} threads"}


def run_reference(args, ws, rank):
    """The reference arm: the plain CPU oracle (there is no other implementation
    of this layer to run), each step a bounded sample of the workload."""
    if rank != 0:
        return None
    import oracle
    from mxfp4_mixture_experts_softmax_gb300 import synth
    if args.steps <= 0:
        args.steps = 50
    w = synth.WORKLOADS[args.workload]
    host = synth.make_inputs(w)
    threads = synth.cpu_threads()
    n = threads  # tokens per step: one per thread

    def step(i):
        ids, wt = oracle.route(host["logits"], w.K, w.with_shared, w.renormalize)
        _oracle_sample(w, host, ids, wt, n, threads, offset=i * n, act=args.act)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    sample = (f"{n} tokens of {w.name} per step (all {w.Kt} experts each) plus routing of the "
              f"{w.T}-token batch, {threads} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)",
        "config": workload_config(w, args.act, ws),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
    else:
        res = run_ours(args, ws, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
