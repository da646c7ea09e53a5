"""Benchmark of the forward MoE layer on one GB300 (replicas on N GPUs).

Workload: the DeepSeek-V3-shaped MXFP8 layer (N=8192 tokens, H=7168, I=2048,
E=256 experts, top-8, 64 virtual source shards of 128 tokens), seeded synthetic
inputs drawn on the device.  One step = one whole forward layer (route + quantise
x, layout, pull dispatch, grouped SwiGLU expert FFN, combine).

Prints one JSON line (rank 0).  `value` is device-timed tokens/s of moe_forward
with inputs resident in HBM; `e2e` is the same call from pinned host buffers with
the host<->device copies inside the timed region; `stages` breaks one step down by
entry point; `roofline` is for the dominant kernel (the expert FFN's two grouped
GEMM launches); `cpu_baseline` times the oracle on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]
                  [--fused]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from token_dispatch_expert_top_gb300 import synth  # noqa: E402

METRIC = "MoE layer fwd tokens/s & TFLOP/s (% MXFP8 peak); dispatch/combine HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0      # nominal dense FP8 / BF16 tensor ratio (4.5 / 2.25 PFLOP/s)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The figure of the slowest rank: all_reduce(MAX) over the process group (any
    backend), the value itself on one rank."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank_step: float, steps: int, t_ms: float, world: int) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank_step * steps / (t_ms / 1e3)


# DRAM bytes (read + write) of one moe_expert_ffn call (its two grouped-GEMM
# launches), from one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum)
# of the 32-expert DeepSeek-V3 stand-in (N=1024, same 256 slots per expert).  The
# full layer has 8x the experts and 8x the slots at the same load per expert, and
# both the weight and the activation bytes grow in proportion, so a full call
# moves 8x that.  Each entry names its capture and the hash of the GEMM sources it
# was taken on (GEMM_SOURCES); a build whose sources hash differently reports no
# traffic, since the counters no longer describe it.
GEMM_SOURCES = ["token_dispatch_expert_top_gb300/csrc/gemm_roles.cuh",
                "token_dispatch_expert_top_gb300/csrc/gemm_tc.cu",
                "token_dispatch_expert_top_gb300/csrc/common.cuh",
                "token_dispatch_expert_top_gb300/csrc/pack.cu"]
FFN_TRAFFIC = {
    "dsv3_mxfp8": {"bytes": 8 * (1.040294 + 0.017880 + 0.501840 + 0.097836) * 1e9,
                   "capture": "profiles/expert_ffn_gemm_dsv3_e32.md", "sources": "a79e2b469015a6d6"},
}


def gemm_sources_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ffn_traffic(workload: str):
    """(bytes per call or None, note) for the expert FFN's two GEMM launches."""
    t = FFN_TRAFFIC.get(workload)
    if t is None:
        return None, "no capture for this workload"
    cur = gemm_sources_hash()
    if cur != t["sources"]:
        return None, f"GEMM sources changed since {t['capture']} (sources {t['sources']}, now {cur})"
    return t["bytes"], f"{t['capture']} (x8 from the 32-expert stand-in; sources {cur})"


def tensor_peak_at(peaks: dict, peak_src: str, dtype: str, clocks: dict):
    """The dense tensor peak for a kernel timed inside the bench's steps: the
    measured burst BF16 GEMM rate (x the nominal FP8/BF16 ratio for MXFP8), scaled
    by the median SM clock sampled during the timed region over the maximum SM clock
    (the burst figure was taken at the maximum clock).  Returns (peak, note)."""
    if dtype == "f32":
        return None, "FP32 SIMT"
    base = peaks["bf16_tflops"] * (FP8_PER_BF16 if dtype == "mxfp8" else 1.0)
    what = f"{peak_src} burst BF16 {peaks['bf16_tflops']:g}" + (
        f" x {FP8_PER_BF16:g} (nominal FP8/BF16)" if dtype == "mxfp8" else "")
    sm, mx = (clocks or {}).get("sm_mhz"), (clocks or {}).get("sm_max_mhz")
    if sm and mx:
        f = min(1.0, sm / mx)
        return base * f, f"{what} x median SM clock {sm:g} / max {mx:g} MHz"
    return base, f"{what} (no clock samples: not scaled)"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ the GPU arm
class StagedStep:
    """The same kernels as moe_forward, issued entry point by entry point so that
    CUDA events can bracket each stage on the launching stream."""

    def __init__(self, layer):
        from token_dispatch_expert_top_gb300 import moe as M
        self.M = M
        self.L = layer
        w = layer.w
        dev = layer.x.device
        T = w.T
        mx = w.dtype == "mxfp8"
        self.mx = mx
        opb = {"f32": 4, "bf16": 2, "mxfp8": 1}[w.dtype]
        self.idx = torch.empty((w.N, w.k), dtype=torch.int32, device=dev)
        self.gate = torch.empty((w.N, w.k), dtype=torch.float32, device=dev)
        self.counts = torch.empty(w.E, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
        self.sched = torch.empty((T, 2), dtype=torch.int32, device=dev)
        self.inv = torch.empty((w.N, w.k), dtype=torch.int32, device=dev)
        if mx:
            self.xq = torch.empty((w.N, w.H), dtype=torch.uint8, device=dev)
            self.xq_sf = torch.empty((w.N, w.H // 32), dtype=torch.uint8, device=dev)
            src, src_sf = self.xq, self.xq_sf
        else:
            self.xq = self.xq_sf = None
            src, src_sf = layer.x, None
        rows = w.rows_per_shard
        self.tab = torch.tensor([src.data_ptr() + s * rows * w.H * opb for s in range(w.S)],
                                dtype=torch.int64, device=dev)
        self.tab_sf = None if not mx else torch.tensor(
            [src_sf.data_ptr() + s * rows * (w.H // 32) for s in range(w.S)], dtype=torch.int64, device=dev)
        self.ring = torch.empty((T, w.H * opb), dtype=torch.uint8, device=dev)
        self.ring_sf = torch.empty((T, w.H // 32), dtype=torch.uint8, device=dev) if mx else None
        self.y = torch.empty((T, w.H), dtype=layer.out.dtype, device=dev)
        self.names = ["route", "layout", "dispatch", "expert_ffn", "combine"]

    def run(self, events=None):
        M, L, w = self.M, self.L, self.L.w
        ev = events or [None] * 6
        if ev[0]:
            ev[0].record()
        M.moe_route_topk(L.x, L.w_router, L.bias, L.shape, self.idx, self.gate, None, self.xq,
                         self.xq_sf, L.ws)
        if ev[1]:
            ev[1].record()
        M.moe_layout(self.idx, L.shape, self.counts, self.offsets, self.sched, self.inv, L.ws)
        if ev[2]:
            ev[2].record()
        M.moe_dispatch_pull(self.tab, self.tab_sf, L.shape, self.sched, self.inv, 0, w.T, self.ring,
                            self.ring_sf, w.T, L.ws)
        if ev[3]:
            ev[3].record()
        M.moe_expert_ffn(self.ring, self.ring_sf, self.offsets, L.wgu, L.wgu_sf, L.wd, L.wd_sf,
                         L.shape, self.y, L.ws)
        if ev[4]:
            ev[4].record()
        M.moe_combine(self.y, self.inv, self.gate, L.shape, L.out, L.ws)
        if ev[5]:
            ev[5].record()


def kernel_launches_per_step(w, fused: bool) -> int:
    """libmoe kernels one forward launches (counted from the launch sequence)."""
    tc_router = w.dtype != "f32" and w.E % 16 == 0 and w.E <= 256 and w.H % 64 == 0
    n = 1 if tc_router else (2 if w.dtype == "mxfp8" else 1)    # router (+ separate x quantiser)
    n += 3                                                      # layout: count, scan, place
    n += 2 if w.dtype == "mxfp8" else 1                         # shard pointer tables
    if fused:
        n += 2                                                  # plan + persistent kernel
    else:
        n += 1 + 2 + 1                                          # dispatch, GEMM1, GEMM2, combine
    return n


def nvfp4_quant_figures(M, x: torch.Tensor, steps: int, hbm: float) -> dict:
    """Time moe_quantize_nvfp4 on the layer's token matrix, L2 flushed before each
    call.  Algorithmic bytes per call: the input read twice (the tensor amax, then
    the blocks) plus the E2M1 codes and E4M3 scales written."""
    rows, K = x.shape
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows, K // 16), dtype=torch.uint8, device=x.device)
    st = torch.empty(2, dtype=torch.float32, device=x.device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=x.device)
    for _ in range(3):
        M.moe_quantize_nvfp4(x, codes, scales, st)
    total = 0.0
    for _ in range(steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        M.moe_quantize_nvfp4(x, codes, scales, st)
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    ms = total / steps
    nbytes = 2 * x.numel() * x.element_size() + codes.numel() + scales.numel()
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"what": f"x [{rows}][{K}] {str(x.dtype).replace('torch.', '')} -> NVFP4 (2 launches)",
            "ms": round(ms, 4), "gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
            "algorithmic_bytes": nbytes, "l2": "flushed (256 MB write) before each call"}


def router_figures(st, steps: int, hbm: float) -> dict:
    """Time moe_route_topk as the layer calls it (x codes and scales written for
    MXFP8), L2 flushed before each call.  Algorithmic bytes per call: x read once,
    W_r read once, the x codes and scales and idx/gate written."""
    M, L, w = st.M, st.L, st.L.w
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=L.x.device)

    def call():
        M.moe_route_topk(L.x, L.w_router, L.bias, L.shape, st.idx, st.gate, None, st.xq, st.xq_sf, L.ws)

    for _ in range(3):
        call()
    total = 0.0
    for _ in range(steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    ms = total / steps
    nbytes = L.x.numel() * L.x.element_size() + L.w_router.numel() * L.w_router.element_size() \
        + st.idx.numel() * 4 + st.gate.numel() * 4
    if st.xq is not None:
        nbytes += st.xq.numel() + st.xq_sf.numel()
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"what": f"moe_route_topk, {w.N} tokens x {w.E} experts, H={w.H}", "ms": round(ms, 4),
            "gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4), "algorithmic_bytes": nbytes,
            "l2": "flushed (256 MB write) before each call"}


def gpu_arm(args, rank, world):
    from token_dispatch_expert_top_gb300 import moe as M
    from token_dispatch_expert_top_gb300.layer import MoeLayer

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w, device=dev)
    layer = MoeLayer(w, inp, device=str(dev))
    del inp
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    rev = M.Params(0, 0, 0, 0, 0, 0, 1) if args.reverse_ring else None

    def fwd(**kw):
        if args.macrobatches > 1:
            return layer.forward_macrobatched(args.macrobatches, x=kw.get("x"), out=kw.get("out"),
                                              stream=kw.get("stream"))
        return layer.forward(fused=args.fused, params=rev, **kw)

    # ---- value: moe_forward (or its macrobatched / fused form), device-resident inputs
    for _ in range(args.warmup):
        fwd()
    status = layer.device_status()
    if status != 0:
        raise RuntimeError(f"device status {M.status_name(status)} after warm-up")
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            fwd()
        ev1.record(stream)
        barrier()
    t_ms = ev0.elapsed_time(ev1)
    status = layer.device_status()
    if status != 0:
        raise RuntimeError(f"device status {M.status_name(status)} in timed region")
    t_ms = max_over_ranks(t_ms, world, dev)
    ms_per_step = t_ms / args.steps
    tokens_per_s = job_rate(w.N, args.steps, t_ms, world)

    # ---- stage breakdown through the individual entry points (same kernels)
    st = StagedStep(layer)
    for _ in range(2):
        st.run()
    torch.cuda.synchronize()
    sums = [0.0] * 5
    for _ in range(args.steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        st.run(evs)
        torch.cuda.synchronize()
        for i in range(5):
            sums[i] += evs[i].elapsed_time(evs[i + 1])
    stage_ms = {n: s / args.steps for n, s in zip(st.names, sums)}
    assert layer.device_status() == 0

    # ---- e2e: the public call from pinned host buffers, copies inside the timed region.
    # Every step copies its x from pinned host memory, runs the layer and reads its
    # out back to pinned host memory.  As a serving loop would, the copies run on
    # their own streams and overlap the layer of the neighbouring step (two device
    # buffers each for x and out); each step's own copies stay inside the region.
    x_host = layer.x.cpu().pin_memory()
    out_host = [torch.empty(layer.out.shape, dtype=layer.out.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(layer.x) for _ in range(2)]
    out_dev = [torch.empty_like(layer.out) for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()

    def e2e_steps(n):
        h2d_done = [ev(), ev()]
        comp_done = [ev(), ev()]
        d2h_done = [None, None]
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(comp_done[b]) if i >= 2 else None   # x_dev[b] free again
                x_dev[b].copy_(x_host, non_blocking=True)
                h2d_done[b].record(s_h2d)
            stream.wait_event(h2d_done[b])
            if d2h_done[b] is not None:
                stream.wait_event(d2h_done[b])                        # out_dev[b] read back
            fwd(x=x_dev[b], out=out_dev[b], stream=stream)
            comp_done[b] = ev()
            comp_done[b].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(comp_done[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                d2h_done[b] = ev()
                d2h_done[b].record(s_d2h)
        for s_ in (s_h2d, s_d2h):
            stream.wait_stream(s_)

    e2e_steps(3)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_h2d.wait_stream(stream)
    s_d2h.wait_stream(stream)
    e2e_steps(args.steps)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    assert torch.equal(out_host[(args.steps - 1) % 2].to(dev), fwd()), "e2e output differs"
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e = {"value": job_rate(w.N, args.steps, e2e_ms, world), "unit": "tokens/s",
           "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
           "d2h_bytes_per_step": out_host[0].numel() * out_host[0].element_size(),
           "overlap": "copies on separate streams, double-buffered device x/out"}

    # ---- derived figures
    peaks, peak_src = load_peaks()
    ffn_flops = w.ffn_flops
    opb = {"f32": 4, "bf16": 2, "mxfp8": 1}[w.dtype]
    row_bytes = w.H * opb + (w.H // 32 if w.dtype == "mxfp8" else 0)
    act = 4 if w.dtype == "f32" else 2
    dispatch_bytes = w.N * row_bytes + w.T * row_bytes
    combine_bytes = w.T * w.H * act + w.N * w.H * act + w.T * 8
    ffn_s = stage_ms["expert_ffn"] / 1e3
    ffn_tflops = ffn_flops / ffn_s / 1e12
    clocks = clk.summary()
    tensor_peak, peak_note = tensor_peak_at(peaks, peak_src, w.dtype, clocks)
    traffic, traffic_note = ffn_traffic(w.name)
    if args.fused:
        # the persistent kernel runs gather + FFN + combine; its time is the step minus
        # the router and layout launches that precede it (same kernels, timed above)
        t_kernel = ms_per_step - stage_ms["route"] - stage_ms["layout"]
        ffn_tflops = ffn_flops / (t_kernel / 1e3) / 1e12
        kname = ("fused persistent kernel (gather + GEMM1/SwiGLU + GEMM2 + combine; time = "
                 "step minus the router and layout launches)")
    else:
        kname = "expert FFN grouped GEMMs (GEMM1+SwiGLU and GEMM2 launches of moe_expert_ffn)"
    roofline = {
        "kernel": kname,
        "bound": "tensor", "achieved": round(ffn_tflops, 2),
        "peak": round(tensor_peak, 1) if tensor_peak else None, "unit": "TFLOP/s",
        "frac": round(ffn_tflops / tensor_peak, 4) if tensor_peak else None,
        "traffic": (None if args.fused else traffic), "traffic_unit": "bytes",
        "traffic_source": "fused kernel: no capture" if args.fused else traffic_note,
        "peak_source": peak_note,
        "algorithmic": f"{ffn_flops / 1e12:.3f} TFLOP per call (6*H*I per slot x {w.T} slots)",
    }
    hbm = peaks["hbm_gbs"]
    disp_gbs = dispatch_bytes / (stage_ms["dispatch"] / 1e3) / 1e9
    comb_gbs = combine_bytes / (stage_ms["combine"] / 1e3) / 1e9
    layer_tflops = world * ffn_flops * args.steps / (t_ms / 1e3) / 1e12
    res = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; x~N(0,1), W~N(0,1/fan_in), drawn on the device)",
        "config": {"workload": w.name, "N": w.N, "H": w.H, "I": w.I, "E": w.E, "k": w.k,
                   "S": w.S, "skew": w.skew,
                   "path": (("fused, reverse ring" if args.reverse_ring else "fused") if args.fused else
                            f"staged, {args.macrobatches} macrobatches" if args.macrobatches > 1 else "staged"),
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: ~11.6 GB of MXFP8 expert weights streamed per step"},
        "layer_tflops": round(layer_tflops, 2),
        "pct_mxfp8_peak_layer": round(layer_tflops / tensor_peak, 4) if tensor_peak else None,
        "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "dispatch_gbs": round(disp_gbs, 1), "dispatch_frac_hbm": round(disp_gbs / hbm, 4),
        "combine_gbs": round(comb_gbs, 1), "combine_frac_hbm": round(comb_gbs / hbm, 4),
        "hbm_peak_gbs": hbm, "hbm_peak_source": peak_src,
        "roofline": roofline,
        "nvfp4_quantize": nvfp4_quant_figures(M, layer.x, args.steps, hbm) if w.dtype != "f32" else None,
        "router": router_figures(st, args.steps, hbm),
        "gpu_launches": kernel_launches_per_step(w, args.fused) * args.steps * max(1, args.macrobatches),
        "clocks": clocks,
        "e2e": e2e,
    }
    if w.skew:
        counts = np.bincount(st.idx.cpu().numpy().ravel(), minlength=w.E)
        res["config"]["load_max_over_mean"] = round(float(counts.max() / counts.mean()), 2)
        res["config"]["empty_experts"] = int((counts == 0).sum())
    if args.ring_sweep:
        res["ring_sweep"] = ring_sweep(M, layer, args)
    return res, layer


def ring_sweep(M, layer, args) -> list:
    """The persistent fused forward over ring sizes of 64, 256 and 1024 slots
    (minibatch = half the ring) and 4, 8 and 16 gather CTAs, each timed with CUDA
    events over --steps steps after 3 warm-up steps, and checked bit for bit
    against the staged forward."""
    sweep = [M.Params(ring, ring // 2, g, 0, 0, 0, 0) for ring in (64, 256, 1024) for g in (4, 8, 16)]
    need = max([M.moe_workspace_bytes(layer.shape, p) for p in sweep] + [layer.ws.numel()])
    if need > layer.ws.numel():                 # one workspace that fits every setting
        layer.ws = torch.empty(need, dtype=torch.uint8, device=layer.out.device)
        M.moe_workspace_init(layer.ws)
    staged = layer.forward().clone()
    rows = []
    for p in sweep:
        for _ in range(3):
            layer.forward(fused=True, params=p)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            out = layer.forward(fused=True, params=p)
        e1.record()
        torch.cuda.synchronize()
        st = layer.device_status()
        rows.append({"ring_slots": p.ring_slots, "minibatch": p.minibatch, "gather_ctas": p.gather_ctas,
                     "ms_per_step": round(e0.elapsed_time(e1) / args.steps, 4),
                     "bitwise_equal_staged": bool(st == 0 and torch.equal(out, staged)),
                     "status": M.status_name(st)})
    return rows


# ------------------------------------------------------------- training step
class BackwardStages:
    """The kernels of moe_backward, issued entry point by entry point so that CUDA
    events can bracket each stage on the launching stream."""

    names = ["reverse_combine", "expert_dgrad", "reverse_dispatch", "router_wgrad", "expert_wgrad"]

    def __init__(self, layer):
        from token_dispatch_expert_top_gb300 import moe as M
        self.M, self.L = M, layer
        w, dev = layer.w, layer.x.device
        mx = w.dtype == "mxfp8"
        T = w.T
        f32 = lambda *s: torch.empty(s, dtype=torch.float32, device=dev)
        bf = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=dev)
        u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device=dev)
        self.dy = u8(T, w.H) if mx else bf(T, w.H)
        self.dy_sf = u8(T, w.H // 32) if mx else None
        self.dgate, self.dlogit, self.sgate, self.sdl = f32(w.N, w.k), f32(w.N, w.k), f32(T), f32(T)
        self.duv = bf(T, 2 * w.I)
        self.duv_c = u8(T, 2 * w.I) if mx else None
        self.duv_s = u8(T, 2 * w.I // 32) if mx else None
        self.da = bf(T, w.H)

    def run(self, dout, events=None):
        M, L, sv = self.M, self.L, self.L.saved
        ev = events or [None] * 6
        rec = lambda i: ev[i].record() if ev[i] else None
        rec(0)
        M.moe_reverse_combine(dout, sv["y"], sv["inv"], sv["gate"], L.shape, self.dy, self.dy_sf,
                              self.dgate, self.dlogit, self.sgate, self.sdl, L.bws)
        rec(1)
        M.moe_expert_ffn_dgrad(self.dy, self.dy_sf, sv["uv"], sv["offsets"], L.wgu_t, L.wgu_t_sf,
                               L.wd_t, L.wd_t_sf, L.shape, self.duv, self.duv_c, self.duv_s, self.da,
                               L.bws)
        rec(2)
        M.moe_reverse_dispatch(self.da, sv["inv"], sv["idx"], self.dlogit, L.w_router, L.shape, L.dx,
                               L.bws)
        rec(3)
        M.moe_router_wgrad(L.x, sv["sched"], sv["offsets"], self.sdl, L.shape, L.dw_router, L.dbias,
                           L.bws)
        rec(4)
        M.moe_expert_wgrad(self.duv, L.x, dout, sv["uv"], sv["sched"], self.sgate, sv["offsets"],
                           L.shape, L.dw_gate_up, L.dw_down, L.bws)
        rec(5)


def train_launches_per_step(w) -> int:
    """libmoe kernels one forward_train + backward launch."""
    fwd = kernel_launches_per_step(w, False)
    bwd = 1 + 2 + 1 + 2 + (1 + 4 + 1)   # rev. combine, dgrad x2, rev. dispatch, router wgrad x2,
    return fwd + bwd                     # wgrad: slot padding, 4 operand packs, GEMM


def train_arm(args, rank, world):
    from token_dispatch_expert_top_gb300 import moe as M
    from token_dispatch_expert_top_gb300.layer import MoeLayer

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w, device=dev)
    layer = MoeLayer(w, inp, device=str(dev), train=True)
    del inp
    gen = torch.Generator(device=dev).manual_seed(w.seed + 7)
    dout = torch.randn((w.N, w.H), generator=gen, device=dev).to(torch.bfloat16)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def step(x=None, g=None):
        layer.forward_train(x=x)
        layer.backward(dout if g is None else g, x=x)

    for _ in range(args.warmup):
        step()
    for st in (layer.device_status(), layer.backward_status()):
        if st != 0:
            raise RuntimeError(f"device status {M.status_name(st)} after warm-up")
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier()
    t_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    assert layer.device_status() == 0 and layer.backward_status() == 0
    ms_per_step = t_ms / args.steps

    # forward time alone (same kernels as forward_train) and the backward stages
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        layer.forward_train()
    f1.record(stream)
    torch.cuda.synchronize()
    fwd_ms = f0.elapsed_time(f1) / args.steps
    bs = BackwardStages(layer)
    bs.run(dout)
    torch.cuda.synchronize()
    sums = [0.0] * 5
    for _ in range(args.steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        bs.run(dout, evs)
        torch.cuda.synchronize()
        for i in range(5):
            sums[i] += evs[i].elapsed_time(evs[i + 1])
    stage_ms = {n: s / args.steps for n, s in zip(bs.names, sums)}
    assert layer.backward_status() == 0

    # e2e: x and dout from pinned host memory, dx back, every step, inside the region
    x_host = layer.x.cpu().pin_memory()
    g_host = dout.cpu().pin_memory()
    dx_host = torch.empty(layer.dx.shape, dtype=layer.dx.dtype).pin_memory()
    x_dev, g_dev = torch.empty_like(layer.x), torch.empty_like(dout)

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        g_dev.copy_(g_host, non_blocking=True)
        step(x_dev, g_dev)
        dx_host.copy_(layer.dx, non_blocking=True)

    for _ in range(2):
        e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e = {"value": job_rate(w.N, args.steps, e2e_ms, world), "unit": "tokens/s",
           "h2d_bytes_per_step": 2 * x_host.numel() * x_host.element_size(),
           "d2h_bytes_per_step": dx_host.numel() * dx_host.element_size(),
           "overlap": "none (copies and the step on one stream)"}

    peaks, peak_src = load_peaks()
    clocks = clk.summary()
    tensor_peak, peak_note = tensor_peak_at(peaks, peak_src, w.dtype, clocks)
    flops = w.ffn_flops                      # each of dgrad and wgrad: 6*H*I per slot
    dgrad_tf = flops / (stage_ms["expert_dgrad"] / 1e3) / 1e12
    wgrad_tf = flops / (stage_ms["expert_wgrad"] / 1e3) / 1e12
    # wgrad writes every expert's BF16 gradients (zeros for idle experts) and reads its
    # inputs once: du|dv (4I B), the x and g*dY rows (2H B each) and u|v (4I B) per slot
    wgrad_bytes = w.E * 3 * w.I * w.H * 2 + w.T * (4 * w.I + 2 * w.H + 2 * w.H + 4 * w.I)
    hbm = peaks["hbm_gbs"]
    dom = "expert_wgrad" if stage_ms["expert_wgrad"] >= stage_ms["expert_dgrad"] else "expert_dgrad"
    if dom == "expert_wgrad" and wgrad_bytes / (hbm * 1e9) > flops / (tensor_peak * 1e12):
        gbs = wgrad_bytes / (stage_ms["expert_wgrad"] / 1e3) / 1e9
        roofline = {
            "kernel": "expert wgrad (slot padding, four operand packs, grouped GEMM)",
            "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(gbs / hbm, 4), "traffic": None, "peak_source": f"{peak_src} copy",
            "algorithmic": (f"{wgrad_bytes / 1e9:.2f} GB per call: BF16 gradients of {w.E} experts "
                            f"(6*I*H B each) + du|dv, x, g*dY and u|v rows read once per slot; "
                            f"the compute floor {flops / (tensor_peak * 1e12) * 1e3:.2f} ms is lower"),
        }
    else:
        dom_tf = wgrad_tf if dom == "expert_wgrad" else dgrad_tf
        roofline = {
            "kernel": ("expert wgrad (slot padding, four operand packs, grouped GEMM)" if dom == "expert_wgrad"
                       else "expert dgrad (two grouped GEMMs and the SwiGLU derivative)"),
            "bound": "tensor", "achieved": round(dom_tf, 2), "peak": round(tensor_peak, 1),
            "unit": "TFLOP/s", "frac": round(dom_tf / tensor_peak, 4), "traffic": None,
            "peak_source": peak_note,
            "algorithmic": f"{flops / 1e12:.3f} TFLOP per call (6*H*I per slot x {w.T} slots)",
        }
    counts = np.bincount(layer.saved["idx"].cpu().numpy().ravel(), minlength=w.E)
    res = {
        "metric": "MoE layer training step (forward + backward) tokens/s", "value":
            round(job_rate(w.N, args.steps, t_ms, world), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; x, dout ~N(0,1), W~N(0,1/fan_in), drawn on the device)",
        "config": {"workload": w.name, "N": w.N, "H": w.H, "I": w.I, "E": w.E, "k": w.k, "S": w.S,
                   "skew": w.skew, "path": "forward_train + backward", "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: ~23 GB of packed MXFP8 weights read per step",
                   "load_max_over_mean": round(float(counts.max() / counts.mean()), 2),
                   "empty_experts": int((counts == 0).sum())},
        "forward_ms": round(fwd_ms, 4),
        "backward_stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "dgrad_tflops": round(dgrad_tf, 2), "dgrad_frac_tensor": round(dgrad_tf / tensor_peak, 4),
        "wgrad_tflops": round(wgrad_tf, 2),
        "roofline": roofline,
        "gpu_launches": train_launches_per_step(w) * args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    return res, layer


# ------------------------------------------------------------- the oracle (CPU)
def oracle_layer_estimate(w, inp, n_experts: int, seed: int):
    """One bounded sample of the forward layer on the oracle, scaled to the whole
    layer.  Timed parts: the router, top-k and layout of all N tokens; the dispatch
    and expert FFN of every slot of n_experts experts drawn at random among those
    with slots (each quantising its own weights, as the layer does once per call);
    the combine and output rounding of min(256, N) tokens.  Returns (estimated
    seconds for the whole layer = route/layout + (experts with slots / n_experts) x
    the sampled experts' time + (N / combined tokens) x the combine time, wall
    seconds spent)."""
    sys.path.insert(0, os.path.join(ROOT, "oracle"))
    import oracle as O

    rng = np.random.default_rng(seed)
    t0 = time.perf_counter()
    x = O._f64(inp["x"])
    logits = O.router_logits(x, inp["w_router"], inp["bias"])
    idx, gate = O.route_topk(logits, w.k)
    counts, offsets, sched, inv = O.layout(idx, w.E, w.S)
    t_route = time.perf_counter() - t0
    live = np.nonzero(counts)[0]
    pick = rng.choice(live, size=min(n_experts, len(live)), replace=False)
    t1 = time.perf_counter()
    fmt_a = O.FORMATS[w.dtype][0]
    for e in pick:
        rows = sched[offsets[e]:offsets[e + 1]]
        tok = rows[:, 0].astype(np.int64) * w.rows_per_shard + rows[:, 1]
        a = x[tok]
        if fmt_a == "mxfp8":
            a = O.mxfp8_values(a)
        wg, wu, wd = O.expert_operands(inp["w_gate_up"][int(e)].cpu(), inp["w_down"][int(e)].cpu(), w.dtype)
        O.expert_ffn(a, wg, wu, wd, w.dtype)
    t_exp = time.perf_counter() - t1
    t2 = time.perf_counter()
    nc = min(256, w.N)
    y = rng.standard_normal((nc * w.k, w.H))
    out = O.combine(y, np.arange(nc * w.k, dtype=np.int32).reshape(nc, w.k), gate[:nc])
    O.round_to(out, O.FORMATS[w.dtype][3])
    t_comb = time.perf_counter() - t2
    est = t_route + t_exp * len(live) / len(pick) + t_comb * w.N / nc
    return est, time.perf_counter() - t0


def oracle_train_sample(w, inp, n_tokens: int, seed: int):
    """One bounded sample of the training step on the oracle: the forward of
    n_tokens sampled tokens (routing and layout of all N) and the backward of
    those tokens' input gradients (their k slots' FFN backward, the gate and
    router terms).  Returns seconds."""
    sys.path.insert(0, os.path.join(ROOT, "oracle"))
    import oracle as O

    toks = np.random.default_rng(seed).choice(w.N, size=n_tokens, replace=False)
    dout = torch.randn((w.N, w.H), generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)

    def weights(e):
        return O.expert_operands(inp["w_gate_up"][e].cpu(), inp["w_down"][e].cpu(), w.dtype)

    t0 = time.perf_counter()
    O.forward({"x": inp["x"], "w_router": inp["w_router"], "bias": inp["bias"]}, w.E, w.k, w.S,
              w.dtype, tokens=toks, weights=weights)
    O.backward({k: inp[k] for k in ("x", "w_router", "bias", "w_gate_up", "w_down")}, w.E, w.k, w.S,
               w.dtype, dout, tokens=toks, experts=[], weights=weights)
    return time.perf_counter() - t0


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    w = synth.WORKLOADS[args.workload]
    dev = "cuda" if (w.name in synth.DEVICE_DRAWN and torch.cuda.is_available()) else "cpu"
    inp = synth.make_inputs(w, device=dev)
    n_exp = args.sample_experts
    est, wall = [], []
    for i in range(args.warmup + args.steps):
        e, t = oracle_layer_estimate(w, inp, n_exp, seed=i)
        if i >= args.warmup:
            est.append(e)
            wall.append(t)
    value = w.N * args.steps / sum(est)
    nc = min(256, w.N)
    sample = (f"per step: routing, top-k and layout of all {w.N} tokens, dispatch + expert FFN of "
              f"every slot of {n_exp} random expert(s) with slots, combine of {nc} tokens (FP64 "
              f"oracle); the layer time is extrapolated from them (experts with slots / {n_exp}, "
              f"N / {nc}); {sum(wall):.1f} s of CPU wall time over {args.steps} steps")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(est) / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "N": w.N, "H": w.H, "I": w.I, "E": w.E, "k": w.k,
                   "S": w.S, "skew": w.skew},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="dsv3_mxfp8", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--fused", action="store_true", help="time moe_forward_fused")
    ap.add_argument("--macrobatches", type=int, default=1,
                    help="time moe_forward_macrobatched with this many macrobatches")
    ap.add_argument("--reverse-ring", action="store_true",
                    help="with --fused: minibatches walk the slots from the last one down")
    ap.add_argument("--sample-tokens", type=int, default=2,
                    help="tokens per oracle sample of the training step's CPU baseline")
    ap.add_argument("--sample-experts", type=int, default=1,
                    help="experts per oracle sample (reference arm; the forward's CPU baseline "
                         "takes at least 16)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--train", action="store_true",
                    help="time the training step (forward_train + backward) instead of the forward")
    ap.add_argument("--ring-sweep", action="store_true",
                    help="also time the fused forward over rings of 64/256/1024 slots x 4/8/16 "
                         "gather CTAs (added to the JSON line as ring_sweep)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group(
            backend="nccl" if args.impl == "gb300" else "gloo")

    if args.impl == "reference":
        res = reference_arm(args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    res, layer = (train_arm if args.train else gpu_arm)(args, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            w = layer.w
            del layer
            torch.cuda.empty_cache()
            inp = synth.make_inputs(w, device="cuda" if w.name in synth.DEVICE_DRAWN else "cpu")
            n_tok = args.sample_tokens
            if args.train:
                dt = oracle_train_sample(w, inp, n_tok, seed=12345)
                what = (f"forward and input-gradient backward of {n_tok} random tokens (routing and "
                        f"layout of all {w.N}), FP64 oracle, {dt:.1f} s")
                value = n_tok / dt
            else:
                n_exp = max(16, args.sample_experts)
                est, dt = oracle_layer_estimate(w, inp, n_exp, seed=12345)
                what = (f"routing, top-k and layout of all {w.N} tokens, dispatch + expert FFN of "
                        f"every slot of {n_exp} random experts with slots, combine of "
                        f"{min(256, w.N)} tokens, "
                        f"FP64 oracle, {dt:.1f} s; the whole layer extrapolated from them: "
                        f"{est:.1f} s")
                value = w.N / est
            res["cpu_baseline"] = {"value": round(value, 4), "unit": "tokens/s",
                                   "cores": cpu_cores(), "kind": "oracle", "sample": what}
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
