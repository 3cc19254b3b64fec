#!/usr/bin/env python3
"""Benchmark of the fused MoE expert layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|skew|kimi|tiny]

A step is one pass of the whole layer (routing, dispatch, L1 GEMM + SwiGLU +
requantisation, L2 GEMM, weighted combine) over one batch of synthetic
inputs.  The default workload is the decode batch: 128 tokens, hidden 7168,
inter 2048 per expert, 256 experts, top-8, FP8-E4M3 activations x FP4-E2M1
weights with UE8M0 scales per 32, clamp 7.  Inputs are synthetic (seeded
generator), resident in HBM before the timed region; the expert weights
(5.9 GB) are far larger than L2, so no flush is needed between steps.

Prints ONE JSON line on stdout (rank 0).  Under torchrun (N > 1) each rank
runs an independent replica on its own GPU with its own tokens ("replicas
only": the single-GPU layer has no exchange step); the timed region is
bracketed by barriers and the max over ranks is reported.

``--impl reference`` times the CPU oracle (the plain fp64 definition) on a
bounded sample of the same workload on the host cores; it is the only other
place this script executes ``oracle/``, besides the ``cpu_baseline`` leg.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "moe_layer_tokens_per_s"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_PER_BF16 = 2.0          # nominal dense rate ratio (4.5 vs 2.25 PFLOP/s)
HBM_TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "megamoe_combine_decode.traffic.json")


# ------------------------------------------------------------------ helpers
def _log(*a):
    print(*a, file=sys.stderr, flush=True)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


KERNEL_SOURCES = ("megamoe.cu", "common.cuh", "numerics.cuh")


def _kernel_source_hash():
    """Hash of the persistent layer kernel's sources (profiles are tied to it)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_expert_layer_idx_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic(workload):
    """DRAM bytes per launch of the layer kernel from the committed ncu summary,
    only if it was taken on the current kernel sources (else None)."""
    try:
        with open(HBM_TRAFFIC_PROFILE) as fh:
            d = json.load(fh)
        if d.get("source_hash") == _kernel_source_hash() and d.get("workload") == workload:
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock and clock-event
    reasons); ``ok`` is False where the library or the device cannot be opened."""

    SM_CLOCK = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid=None, index=0):
        import ctypes

        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            rc = 1
            if uuid:
                rc = self.lib.nvmlDeviceGetHandleByUUID(("GPU-" + str(uuid)).encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
            self.ok = rc == 0
            self.mx = self.clock(max_clock=True)
        except Exception:
            self.ok = False

    def clock(self, max_clock=False):
        import ctypes

        v = ctypes.c_uint(0)
        fn = self.lib.nvmlDeviceGetMaxClockInfo if max_clock else self.lib.nvmlDeviceGetClockInfo
        return v.value if fn(self.h, self.SM_CLOCK, ctypes.byref(v)) == 0 else None

    def reasons(self):
        import ctypes

        v = ctypes.c_ulonglong(0)
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(self.h, ctypes.byref(v)) != 0:
            return None
        return [nm for bit, nm in self.REASONS.items() if v.value & bit]


class ClockSampler:
    """SM clock and throttle reasons sampled DURING the timed region: an NVML
    thread every millisecond (so that even a region of a few tens of
    milliseconds gets tens of samples), else nvidia-smi every 100 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, uuid=None, period_s=0.001):
        self.index, self.uuid, self.period = index, uuid, period_s
        self.proc = None
        self.thread = None
        self.samples = []        # (sm_mhz, [reasons])
        self.max_mhz = None
        self.source = None

    def __enter__(self):
        import threading

        nv = _Nvml(self.uuid, self.index)
        if nv.ok and nv.clock() is not None:
            self.source, self.max_mhz = "nvml", nv.mx
            self._stop = threading.Event()

            def run():
                while not self._stop.is_set():
                    c, r = nv.clock(), nv.reasons()
                    if c is not None:
                        self.samples.append((float(c), r or []))
                    self._stop.wait(self.period)

            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
            return self
        try:
            self.source = "nvidia-smi"
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self._stop.set()
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for ln in out.splitlines():
                f = [x.strip() for x in ln.split(",")]
                if len(f) < 9:
                    continue
                try:
                    c, self.max_mhz = float(f[1]), float(f[2])
                except ValueError:
                    continue
                self.samples.append((c, [nm for nm, v in zip(names, f[5:9]) if v.lower() == "active"]))
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": self.source}
        sm = [c for c, _ in self.samples]
        reasons = sorted({r for _, rs in self.samples for r in rs})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz, "sm_min_mhz": min(sm),
                "reasons": reasons, "samples": len(sm), "source": self.source}


def replica_throughput(ms_local, tokens_per_rank, world, max_over_ranks):
    """Whole-job throughput of `world` independent replicas: every rank ran
    `tokens_per_rank` tokens per step; the job's step time is the slowest
    rank's.  `max_over_ranks(x)` reduces a float across ranks (identity for
    one rank).  Returns (tokens/s, ms per step)."""
    ms = max_over_ranks(ms_local) if world > 1 else ms_local
    return world * tokens_per_rank / (ms * 1e-3), ms


# ------------------------------------------------------------------ our arm
PER_CONFIG = ("prefill", "skew", "kimi")       # timed after the headline in the same run (1 GPU)
PAIR_CONFIG = ("prefill",)                     # also timed with the two-CTA tiles switched on


def _quant(mm, src, rows, cols, fmt, out, out_sf):
    rc = mm.mm_quantize_mx(src, rows, cols, fmt, out, out_sf)
    if rc != mm.MM_OK:
        raise RuntimeError(f"mm_quantize_mx: {mm.STATUS_NAMES.get(rc, rc)}")


def _quant_f8b(mm, src, rows, cols, block_rows, out, out_sf):
    rc = mm.mm_quantize_f8b(src, rows, cols, block_rows, out, out_sf)
    if rc != mm.MM_OK:
        raise RuntimeError(f"mm_quantize_f8b: {mm.STATUS_NAMES.get(rc, rc)}")


def _make_weights(mm, synth, torch, cfg, dev, bf16_layer, f8b=False):
    """Seeded expert weights, quantised on the device by the library's own kernel."""
    E, H, I = cfg.E, cfg.H, cfg.I
    if f8b:
        l1_w = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
        l1_sf = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
        l2_w = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
        l2_sf = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=dev)
    elif bf16_layer:
        l1_w = torch.empty(E, 2 * I, H, dtype=torch.bfloat16, device=dev)
        l2_w = torch.empty(E, H, I, dtype=torch.bfloat16, device=dev)
        l1_sf = l2_sf = None
    else:
        l1_w = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=dev)
        l1_sf = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=dev)
        l2_w = torch.empty(E, H, I // 2, dtype=torch.uint8, device=dev)
        l2_sf = torch.empty(E, H, I // 32, dtype=torch.uint8, device=dev)
    chunk = 16
    buf = torch.empty(min(chunk, E) * 2 * I * H, dtype=torch.float32, device=dev)
    for e0 in range(0, E, chunk):
        e1 = min(E, e0 + chunk)
        n1, n2 = (e1 - e0) * 2 * I * H, (e1 - e0) * H * I
        synth.normal_f32_cuda(cfg.seed, synth.TENSOR_W1, e0 * 2 * I * H, buf[:n1], synth.weight_scale(H))
        if f8b:
            _quant_f8b(mm, buf[:n1], (e1 - e0) * 2 * I, H, 128, l1_w[e0:e1], l1_sf[e0:e1])
        elif bf16_layer:
            l1_w[e0:e1].copy_(buf[:n1].view(e1 - e0, 2 * I, H))
        else:
            _quant(mm, buf[:n1], (e1 - e0) * 2 * I, H, mm.MM_FMT_E2M1, l1_w[e0:e1], l1_sf[e0:e1])
        synth.normal_f32_cuda(cfg.seed, synth.TENSOR_W2, e0 * H * I, buf[:n2], synth.weight_scale(I))
        if f8b:
            _quant_f8b(mm, buf[:n2], (e1 - e0) * H, I, 128, l2_w[e0:e1], l2_sf[e0:e1])
        elif bf16_layer:
            l2_w[e0:e1].copy_(buf[:n2].view(e1 - e0, H, I))
        else:
            _quant(mm, buf[:n2], (e1 - e0) * H, I, mm.MM_FMT_E2M1, l2_w[e0:e1], l2_sf[e0:e1])
    del buf
    if not (f8b or bf16_layer):
        # the one-time transform of the block scales into the layout the layer reads
        l1_sf = mm.prepare_weight_scales(l1_sf, H)
        l2_sf = mm.prepare_weight_scales(l2_sf, I)
    return l1_w, l1_sf, l2_w, l2_sf


def _make_tokens(mm, synth, torch, cfg, seed, dev, bf16_layer, f8b=False):
    T, H = cfg.T, cfg.H
    xf = torch.empty(T * H, dtype=torch.float32, device=dev)
    synth.normal_f32_cuda(seed, synth.TENSOR_X, 0, xf)
    if f8b:
        x = torch.empty(T, H, dtype=torch.uint8, device=dev)
        x_sf = torch.empty(T, H // 128, dtype=torch.float32, device=dev)
        _quant_f8b(mm, xf, T, H, 1, x, x_sf)
    elif bf16_layer:
        x, x_sf = xf.view(T, H).to(torch.bfloat16), None
    else:
        x = torch.empty(T, H, dtype=torch.uint8, device=dev)
        x_sf = torch.empty(T, H // 32, dtype=torch.uint8, device=dev)
        _quant(mm, xf, T, H, mm.MM_FMT_E4M3, x, x_sf)
    del xf
    idx_np, w_np, _ = synth.routing(cfg, seed)
    return x, x_sf, torch.from_numpy(idx_np).to(dev), torch.from_numpy(w_np).to(dev), idx_np


def _roofline(cfg, ms, idx_np, bf16_layer, workload, kernel, route_ms=None, f8b=False):
    """Roofline of one whole step (routing, layer kernel, combine): algorithmic
    bytes (touched experts' weights + scales, x, x_sf, top-k, y) or FLOPs over
    the step time, against the measured peak of the bound that is slower."""
    import numpy as np

    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    counts = np.bincount(idx_np.reshape(-1)[idx_np.reshape(-1) >= 0], minlength=E)
    touched = int((counts > 0).sum())
    if bf16_layer:      # bf16 weights (no scales), bf16 x
        alg_bytes = touched * (3 * H * I * 2) + T * H * 2 + T * k * 8 + T * H * 2
    elif f8b:           # E4M3 weights + fp32 scales per 128 x 128, E4M3 x + fp32 scales per 128
        alg_bytes = touched * (3 * H * I + 3 * (H // 128) * (I // 128) * 4) + T * H + T * (H // 128) * 4 + \
            T * k * 8 + T * H * 2
    else:
        alg_bytes = touched * cfg.expert_bytes() + T * H + T * H // 32 + T * k * 8 + T * H * 2
    hbm, bf16, peak_src = _peaks()
    achieved_gbs = alg_bytes / (ms * 1e-3) / 1e9
    achieved_tflops = cfg.flops() / (ms * 1e-3) / 1e12
    # E4M3 x E2M1 block-scaled MMAs run at the FP8 rate: the measured bf16 peak x the nominal 2
    mx_tflops = bf16 if bf16_layer else FP8_PER_BF16 * bf16
    tensor_bound = cfg.flops() / alg_bytes > (mx_tflops * 1e12) / (hbm * 1e9)
    common = {"peak_source": (f"{peak_src}: MEASURED_PEAKS.json " +
                              (("bf16_tflops" if bf16_layer else "bf16_tflops x 2 (nominal FP8 / bf16)")
                               if tensor_bound else "hbm_gbs"))
              if peak_src == "measured" else "fallback (6.8 TB/s, 1.9 PFLOP/s bf16 x 2)",
              "kernel": kernel, "time_ms": round(ms, 4),
              "algorithmic_bytes_per_launch": alg_bytes, "flops_per_launch": cfg.flops(),
              "touched_experts": touched, "achieved_gbs": round(achieved_gbs, 1),
              "achieved_tflops": round(achieved_tflops, 1),
              "hbm_frac": round(achieved_gbs / hbm, 4), "tensor_frac": round(achieved_tflops / mx_tflops, 4)}
    if route_ms is not None:
        common["route_ms"] = round(route_ms, 4)
    if tensor_bound:
        return {"bound": "tensor", "achieved": round(achieved_tflops, 1), "peak": round(mx_tflops, 1),
                "unit": "TFLOP/s", "frac": round(achieved_tflops / mx_tflops, 4), "traffic": None, **common}
    return {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved_gbs / hbm, 4), "traffic": _profiled_traffic(workload), **common}


def _device_uuid(torch, dev):
    try:
        return str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import moe_expert_layer_idx_gb300 as mm
    import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    uuid = _device_uuid(torch, dev)
    mm.lib()                                           # fails loudly if the library is missing
    cfg = synth.CONFIGS[args.workload]
    seed = cfg.seed + rank                             # replicas: distinct tokens per rank
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    bf16_layer = args.layer == "bf16"
    f8b = args.layer == "f8b"

    # ---- inputs (synthetic, generated and quantised on the device)
    l1_w, l1_sf, l2_w, l2_sf = _make_weights(mm, synth, torch, cfg, dev, bf16_layer, f8b)
    x, x_sf, topk_idx, topk_w, idx_np = _make_tokens(mm, synth, torch, cfg, seed, dev, bf16_layer, f8b)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws_bytes = (mm.mm_bf16_workspace_size if bf16_layer else mm.mm_workspace_size)(T, E, k, H, I)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    def forward_into(x_, x_sf_, idx_, w_, y_):
        if bf16_layer:
            return mm.mm_bf16_forward(T, E, k, H, I, x_, idx_, w_, l1_w, l2_w, y_, cfg.clamp, 0, ws, ws_bytes, stream)
        if f8b:
            return mm.mm_f8b_forward(T, E, k, H, I, x_, x_sf_, idx_, w_, l1_w, l1_sf, l2_w, l2_sf, y_, cfg.clamp,
                                     0, ws, ws_bytes, stream)
        return mm.mm_forward(T, E, k, H, I, x_, x_sf_, idx_, w_, l1_w, l1_sf, l2_w, l2_sf, y_, cfg.clamp, 0,
                             ws, ws_bytes, stream)

    def step():
        rc = forward_into(x, x_sf, topk_idx, topk_w, y)
        if rc != mm.MM_OK:
            raise RuntimeError(f"mm_forward: {mm.STATUS_NAMES.get(rc, rc)}")

    def check_status(w=None):
        st, sm, info = mm.mm_get_status(ws if w is None else w, stream)
        if st != mm.MM_OK:
            raise RuntimeError(f"device status {mm.STATUS_NAMES.get(st, st)} sm={sm} info={info:#x}")

    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        torch.cuda.synchronize(dev)
        if dist:
            tdist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    check_status()

    # ---- timed region: K whole-layer steps, inputs resident
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local_rank, uuid) as clk:
        t_wall = time.perf_counter()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        ev1.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier()
    check_status()
    def max_over_ranks(v):
        t = torch.tensor([v], device=dev, dtype=torch.float64)
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
        return float(t.item())

    tokens_per_s, ms = replica_throughput(ev0.elapsed_time(ev1) / args.steps, T, world, max_over_ranks)

    # ---- per-step distribution (separately, each step between its own events)
    n_pct = max(1, min(args.steps, 100))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_pct)]
    for a_, b_ in evs:
        a_.record(stream)
        step()
        b_.record(stream)
    torch.cuda.synchronize(dev)
    per_step = sorted(a_.elapsed_time(b_) for a_, b_ in evs)
    pct = {"p10": round(float(np.percentile(per_step, 10)), 4), "p50": round(float(np.percentile(per_step, 50)), 4),
           "p90": round(float(np.percentile(per_step, 90)), 4), "steps": n_pct}
    check_status()

    # ---- routing kernel(s) alone: reported beside the whole-step roofline
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(args.steps):
        if mm.mm_route(T, E, k, H, I, topk_idx, ws, ws_bytes, stream) != mm.MM_OK:
            raise RuntimeError("mm_route failed")
    eb.record(stream)
    eb.synchronize()
    route_ms = ea.elapsed_time(eb) / args.steps

    # ---- end to end through the C ABI: pinned host inputs -> device -> layer -> host
    hx = x.cpu().pin_memory()
    hsf = x_sf.cpu().pin_memory() if x_sf is not None else None
    hidx = topk_idx.cpu().pin_memory()
    hw = topk_w.cpu().pin_memory()
    e_steps = max(1, min(args.steps, 200))
    h2d = hx.numel() * hx.element_size() + (hsf.numel() * hsf.element_size() if hsf is not None else 0) + \
        hidx.numel() * 4 + hw.numel() * 4
    d2h = T * H * 2

    def e2e_serial():
        """Every step on one stream: upload, layer, download, one after the other."""
        hy = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()

        def one():
            x.copy_(hx, non_blocking=True)
            if hsf is not None:
                x_sf.copy_(hsf, non_blocking=True)
            topk_idx.copy_(hidx, non_blocking=True)
            topk_w.copy_(hw, non_blocking=True)
            step()
            hy.copy_(y, non_blocking=True)

        for _ in range(2):
            one()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e_steps):
            one()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / e_steps

    def e2e_pipelined():
        """Two sets of device buffers; step i + 1's upload (one copy stream) and step
        i - 1's download (another) overlap step i's layer.  The timed region still
        holds every step's upload, layer and download: it starts before the first
        upload and ends after the last download."""
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        bufs = []
        for _b in range(2):
            bufs.append({"x": torch.empty_like(x), "x_sf": torch.empty_like(x_sf) if x_sf is not None else None,
                         "idx": torch.empty_like(topk_idx), "w": torch.empty_like(topk_w), "y": torch.empty_like(y),
                         "hy": torch.empty(T, H, dtype=torch.bfloat16).pin_memory(),
                         "in": torch.cuda.Event(), "out": torch.cuda.Event(), "d2h": torch.cuda.Event()})
        for bf in bufs:
            bf["out"].record(stream)
            bf["d2h"].record(stream)

        def run(n):
            for i in range(n):
                bf = bufs[i % 2]
                up.wait_event(bf["out"])                  # the layer two steps back has read these inputs
                with torch.cuda.stream(up):
                    bf["x"].copy_(hx, non_blocking=True)
                    if hsf is not None:
                        bf["x_sf"].copy_(hsf, non_blocking=True)
                    bf["idx"].copy_(hidx, non_blocking=True)
                    bf["w"].copy_(hw, non_blocking=True)
                bf["in"].record(up)
                stream.wait_event(bf["in"])
                stream.wait_event(bf["d2h"])              # the download two steps back has read y
                rc = forward_into(bf["x"], bf["x_sf"], bf["idx"], bf["w"], bf["y"])
                if rc != mm.MM_OK:
                    raise RuntimeError(f"forward failed: {mm.STATUS_NAMES.get(rc, rc)}")
                bf["out"].record(stream)
                down.wait_event(bf["out"])
                with torch.cuda.stream(down):
                    bf["hy"].copy_(bf["y"], non_blocking=True)
                bf["d2h"].record(down)
            for bf in bufs:                                # the last downloads end the timed region
                stream.wait_event(bf["d2h"])

        run(2)
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up.wait_event(a)
        run(e_steps)
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / e_steps

    serial_ms = e2e_serial()
    check_status()
    pipe_ms = e2e_pipelined()
    check_status()
    e2e_tps, e2e_ms = replica_throughput(pipe_ms, T, world, max_over_ranks)
    serial_tps, serial_ms = replica_throughput(serial_ms, T, world, max_over_ranks)

    roofline = _roofline(cfg, ms, idx_np, bf16_layer, args.workload,
                         "whole step: routing + megamoe_kernel + combine_kernel", route_ms, f8b)
    roofline["layer_kernel"] = ("f8b (one CTA, 128-token tiles, promotion per 128-K stage)" if f8b else
                                mm.VARIANT_NAMES.get(mm.mm_layer_variant(T, E, k, H, bf16_layer)))
    launches_per_step = (1 if T * k <= 2048 else 3) + 2

    # ---- the other full-size configurations, timed the same way (1 GPU only)
    per_config = {}
    if world == 1 and args.layer == "fp8" and args.per_config:
        del hx, hsf, hidx, hw, ws
        weights = (l1_w, l1_sf, l2_w, l2_sf)
        for name in args.per_config:
            pc = synth.CONFIGS[name]
            if (pc.E, pc.H, pc.I) != (E, H, I):
                weights = None
                del l1_w, l1_sf, l2_w, l2_sf
                torch.cuda.empty_cache()
                l1_w, l1_sf, l2_w, l2_sf = _make_weights(mm, synth, torch, pc, dev, False)
                weights = (l1_w, l1_sf, l2_w, l2_sf)
                E, H, I = pc.E, pc.H, pc.I
            runs = [(name, None)] + ([(f"{name} (two-CTA tiles)", 1)] if name in args.pair_config else [])
            for key, pair in runs:
                prev = mm.mm_set_pair_mma(pair) if pair is not None else None
                try:
                    per_config[key] = _time_config(mm, synth, torch, np, pc, weights, dev, stream, uuid, local_rank,
                                                   args.per_config_steps, max(3, args.warmup))
                finally:
                    if prev is not None:
                        mm.mm_set_pair_mma(prev)
                per_config[key]["layer_kernel"] = mm.VARIANT_NAMES.get(
                    mm.mm_layer_variant(pc.T, pc.E, pc.k, pc.H) if pair is None else 4)
                launches_per_step_pc = (1 if pc.T * pc.k <= 2048 else 3) + 2
                per_config[key]["gpu_launches"] = launches_per_step_pc * per_config[key]["steps"]
    return {
        "tokens_per_s": tokens_per_s, "ms": ms, "route_ms": route_ms, "roofline": roofline,
        "e2e": {"value": round(e2e_tps, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "copies": "two copy streams: step i+1's upload and step i-1's download overlap step i's layer",
                "serial": {"value": round(serial_tps, 1), "ms_per_step": round(serial_ms, 4),
                           "copies": "upload, layer, download in order on one stream"}},
        "clocks": clk.summary(), "wall_s": t_wall, "gpu_launches": launches_per_step * args.steps, "step_ms": pct,
        "cfg": cfg, "per_config": per_config,
    }


def _time_config(mm, synth, torch, np, cfg, weights, dev, stream, uuid, local_rank, steps, warmup):
    """One full-size configuration: W warm-up steps, then K steps between CUDA
    events on the launching stream with the clocks sampled meanwhile; the
    roofline of the whole step.  The expert weights are resident (several GB,
    far beyond L2), so no flush is needed."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    l1_w, l1_sf, l2_w, l2_sf = weights
    x, x_sf, topk_idx, topk_w, idx_np = _make_tokens(mm, synth, torch, cfg, cfg.seed, dev, False)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws_bytes = mm.mm_workspace_size(T, E, k, H, I)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def step():
        rc = mm.mm_forward(T, E, k, H, I, x, x_sf, topk_idx, topk_w, l1_w, l1_sf, l2_w, l2_sf, y, cfg.clamp, 0,
                           ws, ws_bytes, stream)
        if rc != mm.MM_OK:
            raise RuntimeError(f"mm_forward ({cfg.name}): {mm.STATUS_NAMES.get(rc, rc)}")

    for _ in range(warmup):
        step()
    st, sm, info = mm.mm_get_status(ws, stream)
    if st != mm.MM_OK:
        raise RuntimeError(f"{cfg.name}: device status {mm.STATUS_NAMES.get(st, st)} sm={sm} info={info:#x}")
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank, uuid) as clk:
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        ev1.synchronize()
    st, sm, info = mm.mm_get_status(ws, stream)
    if st != mm.MM_OK:
        raise RuntimeError(f"{cfg.name}: device status {mm.STATUS_NAMES.get(st, st)} sm={sm} info={info:#x}")
    ms = ev0.elapsed_time(ev1) / steps
    out = {"workload": f"{cfg.name}: {T} tokens, hidden {H}, inter {I}, {E} experts, top-{k}, "
                       f"E4M3 x E2M1 with UE8M0/32, clamp {cfg.clamp if cfg.clamp else 'none'}",
           "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 4), "tokens_per_s": round(T / (ms * 1e-3), 1),
           "roofline": _roofline(cfg, ms, idx_np, False, cfg.name,
                                 "whole step: routing + megamoe_kernel + combine_kernel"),
           "clocks": clk.summary()}
    if cfg.name == "kimi":
        out["note"] = ("default reserve of 2 SMs, no side stream; the side-stream and graph-replay runs of this "
                       "configuration are parity tests")
    del x, x_sf, topk_idx, topk_w, y, ws
    return out


# ------------------------------------------------------------------ oracle
def _oracle_sample(workload, sample_tokens, layer="fp8"):
    """Prepare a bounded sample of the workload for the CPU oracle (fp64, plain
    numpy): the first `sample_tokens` tokens and the experts they touch (expert
    weights quantised by the oracle).  Returns (run, description, threads)
    where run() is one oracle forward over the sample."""
    import synth
    from oracle import formats as OF
    from oracle import moe as OM
    from oracle import moe_bf16 as OMB
    from oracle import moe_f8b as OM8

    cfg = synth.CONFIGS[workload]
    idx, w, _ = synth.routing(cfg)
    toks = list(range(min(max(1, sample_tokens), cfg.T)))
    experts = sorted({int(e) for e in idx[toks].reshape(-1) if e >= 0})
    tp = time.perf_counter()
    if layer == "f8b":
        xc, xsf = OM8.quantize_tokens_f8b(synth.x_f32(cfg, rows=toks))
        cache = {e: OM8.quantize_expert_f8b(synth.w1_f32(cfg, e), synth.w2_f32(cfg, e)) for e in experts}
        run = lambda: OM8.moe_forward_f8b(xc, xsf, idx[toks], w[toks], lambda e: cache[e], cfg.clamp, cfg.E)  # noqa: E731
    elif layer == "bf16":
        xb = OF.bf16_round(synth.x_f32(cfg, rows=toks))
        cache = {e: (OF.bf16_round(synth.w1_f32(cfg, e)), OF.bf16_round(synth.w2_f32(cfg, e))) for e in experts}
        run = lambda: OMB.moe_forward_bf16(xb, idx[toks], w[toks], lambda e: cache[e], cfg.clamp, cfg.E)  # noqa: E731
    else:
        xc, xsf = OF.quantize_mx(synth.x_f32(cfg, rows=toks), OF.E4M3)
        cache = {e: OM.quantize_expert(synth.w1_f32(cfg, e), synth.w2_f32(cfg, e)) for e in experts}
        run = lambda: OM.moe_forward(xc, xsf, idx[toks], w[toks], lambda e: cache[e], cfg.clamp, cfg.E)  # noqa: E731
    _log(f"oracle sample: {len(experts)} experts prepared in {time.perf_counter() - tp:.1f} s")
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"first {len(toks)} token(s) of the {workload} batch ({len(experts)} experts, "
            f"{len(toks) * cfg.k} assignments); fp64 numpy oracle, BLAS threads default")
    return run, desc, threads, len(toks)


def run_oracle_sample(workload, sample_tokens, layer="fp8"):
    """Time one oracle forward over the sample.  Returns (tokens/s, threads,
    sample description, seconds)."""
    run, desc, threads, n = _oracle_sample(workload, sample_tokens, layer)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    return n / dt, threads, desc, dt


def run_reference(args, config):
    """The reference arm: the oracle, as it stands, on the host cores.  Every
    step is one oracle forward over the same bounded sample of the workload;
    W untimed warm-up steps, then exactly K timed steps."""
    run, desc, threads, n = _oracle_sample(args.workload, args.ref_sample_tokens, args.layer)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    ms = 1e3 * dt / args.steps
    tps = n / (ms * 1e-3)
    return {"impl": "reference", "metric": METRIC, "value": round(tps, 4), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": round(tps, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"each step: {desc}", "tokens_per_step": n,
                             "timed_seconds": round(dt, 2)},
            "e2e": {"value": round(tps, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--layer", choices=["fp8", "bf16", "f8b"], default="fp8",
                    help="fp8: E4M3 x E2M1 with UE8M0/32 (the default); bf16: the bf16 x bf16 layer; "
                         "f8b: the (1, 128, 128) recipe (E4M3 x E4M3, fp32 scales per 1x128 / 128x128)")
    ap.add_argument("--cpu-sample-tokens", type=int, default=8)
    ap.add_argument("--ref-sample-tokens", type=int, default=1,
                    help="tokens per step of the reference arm (the oracle)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-config", default=",".join(PER_CONFIG),
                    help="full-size configurations timed after the headline (1 GPU); empty for none")
    ap.add_argument("--per-config-steps", type=int, default=20)
    ap.add_argument("--pair-config", default=",".join(PAIR_CONFIG),
                    help="per-config workloads also timed with the two-CTA tiles switched on")
    ap.add_argument("--tokens", type=int, default=0, help="override the token count (profiling of small cases)")
    ap.add_argument("--experts", type=int, default=0, help="override the expert count (profiling of small cases)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.per_config = [c for c in args.per_config.split(",") if c and c != args.workload]
    args.pair_config = [c for c in args.pair_config.split(",") if c]

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    import dataclasses

    import synth

    cfg = synth.CONFIGS[args.workload]
    if args.tokens or args.experts:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}-T{args.tokens or cfg.T}-E{args.experts or cfg.E}",
                                  T=args.tokens or cfg.T, E=args.experts or cfg.E)
        synth.CONFIGS[cfg.name] = cfg
        args.workload = cfg.name
        args.per_config = []
    config = {"workload": f"{cfg.name}: {cfg.T} tokens, hidden {cfg.H}, inter {cfg.I}, {cfg.E} experts, "
                          f"top-{cfg.k}, "
                          f"{ {'bf16': 'bf16 x bf16', 'f8b': 'E4M3 x E4M3 with fp32 scales per 1x128 / 128x128'}.get(args.layer, 'E4M3 x E2M1 with UE8M0/32')}, "
                          f"clamp {cfg.clamp if cfg.clamp else 'none'}",
              "tokens": cfg.T, "hidden": cfg.H, "inter": cfg.I, "experts": cfg.E, "topk": cfg.k,
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
              "l2": "inputs larger than L2 (expert weights far exceed 129 MB); no flush"}

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, config)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as tdist

        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    res = run_ours(args, rank, world, local_rank)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            tps, threads, desc, dt = run_oracle_sample(args.workload, args.cpu_sample_tokens, layer=args.layer)
            cpu = {"value": round(tps, 4), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
                   "seconds": round(dt, 2)}
        except Exception as exc:  # the baseline must never hide the GPU number
            cpu = {"value": None, "unit": UNIT, "cores": None, "kind": "oracle", "sample": f"failed: {exc}"}
    if world > 1:
        import torch.distributed as tdist

        tdist.barrier()
        tdist.destroy_process_group()
    if rank != 0:
        return 0
    line = {"metric": METRIC, "value": round(res["tokens_per_s"], 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms"], 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16xbf16->f32", "f8b": "e4m3xe4m3->f32"}.get(args.layer, "e4m3xe2m1->f32"),
            "data": "synthetic", "config": config, "roofline": res["roofline"], "cpu_baseline": cpu,
            "e2e": res["e2e"], "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
            "route_ms": round(res["route_ms"], 4), "step_ms_percentiles": res["step_ms"]}
    if res["per_config"]:
        line["per_config"] = res["per_config"]
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
