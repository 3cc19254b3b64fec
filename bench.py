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


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def replica_throughput(ms_local, tokens_per_rank, world, max_over_ranks):
    """Whole-job throughput of `world` independent replicas: every rank ran
    `tokens_per_rank` tokens per step; the job's step time is the slowest
    rank's.  `max_over_ranks(x)` reduces a float across ranks (identity for
    one rank).  Returns (tokens/s, ms per step)."""
    ms = max_over_ranks(ms_local) if world > 1 else ms_local
    return world * tokens_per_rank / (ms * 1e-3), ms


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import moe_expert_layer_idx_gb300 as mm
    import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    mm.lib()                                           # fails loudly if the library is missing
    cfg = synth.CONFIGS[args.workload]
    seed = cfg.seed + rank                             # replicas: distinct tokens per rank
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k

    # ---- inputs (synthetic, generated and quantised on the device)
    def quant(src, rows, cols, fmt, out, out_sf):
        rc = mm.mm_quantize_mx(src, rows, cols, fmt, out, out_sf)
        if rc != mm.MM_OK:
            raise RuntimeError(f"mm_quantize_mx: {mm.STATUS_NAMES.get(rc, rc)}")

    bf16_layer = args.layer == "bf16"
    if bf16_layer:
        # the bf16 x bf16 layer: the same seeded values, rounded to bf16
        l1_w = torch.empty(E, 2 * I, H, dtype=torch.bfloat16, device=dev)
        l2_w = torch.empty(E, H, I, dtype=torch.bfloat16, device=dev)
        l1_sf = l2_sf = x_sf = None
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
        if bf16_layer:
            l1_w[e0:e1].copy_(buf[:n1].view(e1 - e0, 2 * I, H))
        else:
            quant(buf[:n1], (e1 - e0) * 2 * I, H, mm.MM_FMT_E2M1, l1_w[e0:e1], l1_sf[e0:e1])
        synth.normal_f32_cuda(cfg.seed, synth.TENSOR_W2, e0 * H * I, buf[:n2], synth.weight_scale(I))
        if bf16_layer:
            l2_w[e0:e1].copy_(buf[:n2].view(e1 - e0, H, I))
        else:
            quant(buf[:n2], (e1 - e0) * H, I, mm.MM_FMT_E2M1, l2_w[e0:e1], l2_sf[e0:e1])
    del buf
    xf = torch.empty(T * H, dtype=torch.float32, device=dev)
    synth.normal_f32_cuda(seed, synth.TENSOR_X, 0, xf)
    if bf16_layer:
        x = xf.view(T, H).to(torch.bfloat16)
    else:
        x = torch.empty(T, H, dtype=torch.uint8, device=dev)
        x_sf = torch.empty(T, H // 32, dtype=torch.uint8, device=dev)
        quant(xf, T, H, mm.MM_FMT_E4M3, x, x_sf)
    del xf
    idx_np, w_np, _ = synth.routing(cfg, seed)
    topk_idx = torch.from_numpy(idx_np).to(dev)
    topk_w = torch.from_numpy(w_np).to(dev)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws_bytes = (mm.mm_bf16_workspace_size if bf16_layer else mm.mm_workspace_size)(T, E, k, H, I)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    def step():
        if bf16_layer:
            rc = mm.mm_bf16_forward(T, E, k, H, I, x, topk_idx, topk_w, l1_w, l2_w, y, cfg.clamp, 0, ws, ws_bytes,
                                    stream)
        else:
            rc = mm.mm_forward(T, E, k, H, I, x, x_sf, topk_idx, topk_w, l1_w, l1_sf, l2_w, l2_sf, y, cfg.clamp, 0,
                               ws, ws_bytes, stream)
        if rc != mm.MM_OK:
            raise RuntimeError(f"mm_forward: {mm.STATUS_NAMES.get(rc, rc)}")

    def check_status():
        st, sm, info = mm.mm_get_status(ws, stream)
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
    with ClockSampler(local_rank) as clk:
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

    # ---- routing kernel alone (to isolate the time of the layer kernel and its combine kernel)
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(args.steps):
        if mm.mm_route(T, E, k, H, I, topk_idx, ws, ws_bytes, stream) != mm.MM_OK:
            raise RuntimeError("mm_route failed")
    eb.record(stream)
    eb.synchronize()
    route_ms = ea.elapsed_time(eb) / args.steps
    kernel_ms = max(ms - route_ms, 1e-6)

    # ---- end to end through the C ABI: pinned host inputs -> device -> layer -> host
    hx = x.cpu().pin_memory()
    hsf = x_sf.cpu().pin_memory() if x_sf is not None else None
    hidx = topk_idx.cpu().pin_memory()
    hw = topk_w.cpu().pin_memory()
    hy = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    e_steps = max(1, min(args.steps, 200))

    def e2e_step():
        x.copy_(hx, non_blocking=True)
        if hsf is not None:
            x_sf.copy_(hsf, non_blocking=True)
        topk_idx.copy_(hidx, non_blocking=True)
        topk_w.copy_(hw, non_blocking=True)
        step()
        hy.copy_(y, non_blocking=True)

    for _ in range(2):
        e2e_step()
    barrier()
    e0_, e1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0_.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1_.record(stream)
    e1_.synchronize()
    check_status()
    e2e_tps, e2e_ms = replica_throughput(e0_.elapsed_time(e1_) / e_steps, T, world, max_over_ranks)
    h2d = hx.numel() * hx.element_size() + (hsf.numel() if hsf is not None else 0) + hidx.numel() * 4 + hw.numel() * 4
    d2h = hy.numel() * 2

    # ---- roofline of the layer kernel (HBM-bound at the decode batch)
    counts = np.bincount(idx_np.reshape(-1)[idx_np.reshape(-1) >= 0], minlength=E)
    touched = int((counts > 0).sum())
    if bf16_layer:      # bf16 weights (no scales), bf16 x
        alg_bytes = touched * (3 * H * I * 2) + T * H * 2 + T * k * 8 + T * H * 2
    else:
        alg_bytes = (touched * cfg.expert_bytes() + T * H + T * H // 32 + T * k * 8 + T * H * 2)
    hbm, bf16, peak_src = _peaks()
    achieved_gbs = alg_bytes / (kernel_ms * 1e-3) / 1e9
    achieved_tflops = cfg.flops() / (kernel_ms * 1e-3) / 1e12
    # E4M3 x E2M1 block-scaled MMAs run at the FP8 rate: the measured bf16 peak x the nominal 2
    mx_tflops = bf16 if bf16_layer else FP8_PER_BF16 * bf16
    tensor_bound = cfg.flops() / alg_bytes > (mx_tflops * 1e12) / (hbm * 1e9)
    common = {"peak_source": (f"{peak_src}: MEASURED_PEAKS.json " +
                              (("bf16_tflops" if bf16_layer else "bf16_tflops x 2 (nominal FP8 / bf16)")
                               if tensor_bound else "hbm_gbs"))
              if peak_src == "measured" else "fallback (6.8 TB/s, 1.9 PFLOP/s bf16 x 2)",
              "kernel": "megamoe_kernel + combine_kernel", "kernel_ms": round(kernel_ms, 4),
              "algorithmic_bytes_per_launch": alg_bytes, "flops_per_launch": cfg.flops(),
              "touched_experts": touched, "achieved_gbs": round(achieved_gbs, 1),
              "achieved_tflops": round(achieved_tflops, 1)}
    if tensor_bound:
        roofline = {"bound": "tensor", "achieved": round(achieved_tflops, 1), "peak": round(mx_tflops, 1),
                    "unit": "TFLOP/s", "frac": round(achieved_tflops / mx_tflops, 4), "traffic": None, **common}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(achieved_gbs / hbm, 4), "traffic": _profiled_traffic(args.workload), **common}
    return {
        "tokens_per_s": tokens_per_s, "ms": ms, "route_ms": route_ms, "roofline": roofline,
        "e2e": {"value": round(e2e_tps, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "clocks": clk.summary(), "wall_s": t_wall, "gpu_launches": ((1 if T * k <= 2048 else 3) + 2) * args.steps, "step_ms": pct,
        "cfg": cfg, "touched": touched,
    }


# ------------------------------------------------------------------ oracle
def run_oracle_sample(workload, sample_tokens, time_budget_s=25.0, layer="fp8"):
    """Time the CPU oracle (fp64, plain numpy) on the first tokens of the same
    workload.  Returns (tokens/s, threads, sample description)."""
    import numpy as np

    import synth
    from oracle import formats as OF
    from oracle import moe as OM
    from oracle import moe_bf16 as OMB

    cfg = synth.CONFIGS[workload]
    idx, w, _ = synth.routing(cfg)
    n = max(1, sample_tokens)
    toks = list(range(min(n, cfg.T)))
    experts = sorted({int(e) for e in idx[toks].reshape(-1) if e >= 0})
    tp = time.perf_counter()
    if layer == "bf16":
        xb = OF.bf16_round(synth.x_f32(cfg, rows=toks))
        cache = {e: (OF.bf16_round(synth.w1_f32(cfg, e)), OF.bf16_round(synth.w2_f32(cfg, e))) for e in experts}
    else:
        xc, xsf = OF.quantize_mx(synth.x_f32(cfg, rows=toks), OF.E4M3)
        cache = {e: OM.quantize_expert(synth.w1_f32(cfg, e), synth.w2_f32(cfg, e)) for e in experts}
    _log(f"oracle sample: {len(experts)} experts prepared in {time.perf_counter() - tp:.1f} s")
    t0 = time.perf_counter()
    if layer == "bf16":
        OMB.moe_forward_bf16(xb, idx[toks], w[toks], lambda e: cache[e], cfg.clamp, cfg.E)
    else:
        OM.moe_forward(xc, xsf, idx[toks], w[toks], lambda e: cache[e], cfg.clamp, cfg.E)
    dt = time.perf_counter() - t0
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"first {len(toks)} token(s) of the {workload} batch ({len(experts)} experts, "
            f"{len(toks) * cfg.k} assignments); fp64 numpy oracle, BLAS threads default")
    return len(toks) / dt, threads, desc, dt


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--layer", choices=["fp8", "bf16"], default="fp8",
                    help="fp8: E4M3 x E2M1 (the default); bf16: the bf16 x bf16 layer")
    ap.add_argument("--cpu-sample-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="override the token count (profiling of small cases)")
    ap.add_argument("--experts", type=int, default=0, help="override the expert count (profiling of small cases)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

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
    config = {"workload": f"{cfg.name}: {cfg.T} tokens, hidden {cfg.H}, inter {cfg.I}, {cfg.E} experts, "
                          f"top-{cfg.k}, "
                          f"{'bf16 x bf16' if args.layer == 'bf16' else 'E4M3 x E2M1 with UE8M0/32'}, "
                          f"clamp {cfg.clamp if cfg.clamp else 'none'}",
              "tokens": cfg.T, "hidden": cfg.H, "inter": cfg.I, "experts": cfg.E, "topk": cfg.k,
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
              "l2": "inputs larger than L2 (expert weights far exceed 129 MB); no flush"}

    if args.impl == "reference":
        if rank != 0:
            return 0
        tps, threads, desc, dt = run_oracle_sample(args.workload, args.cpu_sample_tokens, layer=args.layer)
        line = {"impl": "reference", "metric": METRIC, "value": round(tps, 4), "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * cfg.T / tps, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": round(tps, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": round(tps, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
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
            "dtype": "bf16xbf16->f32" if args.layer == "bf16" else "e4m3xe2m1->f32",
            "data": "synthetic", "config": config, "roofline": res["roofline"], "cpu_baseline": cpu,
            "e2e": res["e2e"], "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
            "route_ms": round(res["route_ms"], 4), "step_ms_percentiles": res["step_ms"]}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
