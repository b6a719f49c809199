"""Benchmark: qwen3moe MoE-FFN tokens/s/layer and expert-weight HBM GB/s on GB300.

Workload: one Qwen3-30B-A3B MoE layer at decode (hidden 2048, 128 experts,
top-8 renormalised, expert FFN 768, one token, Q4_K gate/up, Q6_K down),
seeded synthetic weights.  A step is one full MoE-FFN layer call for one token
(router, top-k, per-expert pair lists, gate/up + SwiGLU, down, weighted
combine into the residual) through the C ABI.

Timing: W warm-up steps, then exactly K steps replayed from CUDA graphs,
bracketed by a barrier and a device synchronise, timed with CUDA events on the
launching stream.  Every step reads a different device copy of the layer's
weights; the copies rotate over more than 4x the L2 size, so weight bytes come
from HBM.  ``value`` = tokens/s/layer summed over ranks (each rank runs its own
replica; weak scaling).

``--impl reference`` times the CPU oracle (the reference arm of this repo) on
the same workload and unit.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD_CFG = 2
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copies", type=int, default=32, help="weight copies in the rotation")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            hbm = j.get("hbm_gbs") or j.get("hbm_GBps")
            if hbm:
                return float(hbm), "measured", j
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback", None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (ts, l) in self.lines if t0 - 0.15 <= ts <= t1 + 0.15] or \
            [l for (_, l) in self.lines]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(mx)) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes(inp, ids) -> dict:
    """Bytes the method must read: the distinct selected experts' gate+up+down slices."""
    H, F = inp["H"], inp["F"]
    per = (synth.matrix_bytes(inp["gate_t"], F, H) + synth.matrix_bytes(inp["up_t"], F, H)
           + synth.matrix_bytes(inp["down_t"], H, F))
    distinct = len(np.unique(ids))
    return dict(expert=distinct * per, router=inp["E"] * H * 4,
                act=inp["T"] * H * 4 * 2, distinct=distinct)


def cpu_baseline(inp, seconds: float) -> dict:
    import oracle
    oracle.build()
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    one = dict(inp)
    done, t0 = 0, time.perf_counter()
    rng = np.random.default_rng(123)
    while True:
        one["x"] = rng.standard_normal((1, inp["H"])).astype(np.float32)
        oracle.moe_forward(one)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds and done >= 3:
            break
    return {"value": done / el, "unit": "tokens/s/layer", "cores": cores, "kind": "oracle",
            "sample": f"{done} single-token MoE-FFN layer calls of the decode workload "
                      f"(router + top-8 + 8 experts in double), {el:.1f} s"}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        pg = dist
    return ws, rank, local, pg


def run_reference(args):
    ws, rank, local, pg = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0, None
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cfg = synth.MOE_CONFIGS[WORKLOAD_CFG]
    inp = synth.moe_inputs(cfg)
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    rng = np.random.default_rng(7)
    xs = [rng.standard_normal((1, inp["H"])).astype(np.float32) for _ in range(8)]

    def step(i):
        one = dict(inp)
        one["x"] = xs[i % len(xs)]
        oracle.moe_forward(one)

    t0 = time.perf_counter()
    step(0)
    est = time.perf_counter() - t0
    warm = min(args.warmup, 2)
    for i in range(warm):
        step(i)
    budget = 150.0
    k = max(3, min(args.steps, int(budget / max(est, 1e-6))))
    t0 = time.perf_counter()
    for i in range(k):
        step(i)
    el = time.perf_counter() - t0
    val = k / el
    line = {"impl": "reference", "metric": "qwen3moe MoE-FFN tokens/s/layer", "value": val,
            "unit": "tokens/s/layer", "n_gpus": args.gpus, "steps": k, "requested_steps": args.steps,
            "warmup": warm, "ms_per_step": 1000 * el / k, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "qwen3moe-30b-a3b MoE layer decode, T=1, Q4_K gate/up, Q6_K down",
                       "hidden": 2048, "n_experts": 128, "top_k": 8, "ffn": 768, "tokens": 1},
            "cpu_baseline": {"value": val, "unit": "tokens/s/layer", "cores": cores,
                             "kind": "oracle",
                             "sample": f"{k} single-token layer calls (steps capped to ~{budget:.0f} s)"},
            "e2e": {"value": val, "unit": "tokens/s/layer", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    ws, rank, local, pg = dist_init()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    import quantized_mixture_experts_f32_gb300 as q

    cfg = synth.MOE_CONFIGS[WORKLOAD_CFG]
    inp = synth.moe_inputs(cfg)
    T, H, E, K, F = inp["T"], inp["H"], inp["E"], inp["K"], inp["F"]
    gt, ut, dt = q.QTYPE[inp["gate_t"]], q.QTYPE[inp["up_t"]], q.QTYPE[inp["down_t"]]
    x = torch.from_numpy(inp["x"]).to(dev)
    base = {n: torch.from_numpy(np.ascontiguousarray(inp[n])).to(dev)
            for n in ("router", "gate", "up", "down")}
    R = args.copies
    copies = [base] + [{n: t.clone() for n, t in base.items()} for _ in range(R - 1)]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    ctx = q.qmoe_create(q.make_config(H, E, K, F, T, 1, stream.cuda_stream))

    def call(c):
        q.qmoe_forward(ctx, x, c["router"], c["gate"], c["up"], c["down"], gt, ut, dt, T, out)

    # routing of this input (same for every copy): for the algorithmic bytes
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        q.qmoe_forward_ex(ctx, x, None, None, base["router"], base["gate"], base["up"],
                          base["down"], gt, ut, dt, T, out, ids, None)
    stream.synchronize()
    ab = algorithmic_bytes(inp, ids.cpu().numpy())
    touched = (ab["expert"] + ab["router"]) * R

    with torch.cuda.stream(stream):
        for i in range(3):
            call(copies[i % R])
        stream.synchronize()
        g_full = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_full, stream=stream):
            for i in range(R):
                call(copies[i])
        rem = args.steps % R
        g_rem = None
        if rem:
            g_rem = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_rem, stream=stream):
                for i in range(rem):
                    call(copies[i])
        # warm-up: W steps
        for _ in range(args.warmup // R):
            g_full.replay()
        for i in range(args.warmup % R):
            call(copies[i])
        stream.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps // R):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    stream.synchronize()
    t1 = time.time()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    clocks = sampler.stop(t0, t1)
    ms = e0.elapsed_time(e1)
    if pg:
        tt = torch.tensor([ms], device=dev)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        ms = float(tt.item())
    secs = ms / 1e3
    tokens = T * args.steps * ws
    value = tokens / secs
    step_s = secs / args.steps
    gbs = ab["expert"] / step_s / 1e9

    # e2e: the public host-buffer entry point, copies + sync inside every step
    hin = torch.from_numpy(inp["x"].copy()).pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    for i in range(5):
        q.qmoe_forward_host(ctx, hin, copies[i % R]["router"], copies[i % R]["gate"],
                            copies[i % R]["up"], copies[i % R]["down"], gt, ut, dt, T, hout)
    if pg:
        pg.barrier()
    te0 = time.perf_counter()
    for i in range(args.e2e_steps):
        c = copies[i % R]
        q.qmoe_forward_host(ctx, hin, c["router"], c["gate"], c["up"], c["down"], gt, ut, dt, T,
                            hout)
    te = time.perf_counter() - te0
    if pg:
        tt = torch.tensor([te], device=dev)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        te = float(tt.item())
    e2e_val = T * args.e2e_steps * ws / te

    peak, peak_kind, _ = peaks()
    roof = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "peak_kind": peak_kind, "traffic": None,
            "kernel": "whole MoE-FFN layer call (all kernels of one step)",
            "algorithmic_bytes_per_launch": ab["expert"]}
    line = {
        "metric": "qwen3moe MoE-FFN tokens/s/layer; expert-weight HBM GB/s vs GB300 peak",
        "value": value, "unit": "tokens/s/layer", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "qwen3moe-30b-a3b MoE layer decode, T=1, Q4_K gate/up, Q6_K down",
                   "hidden": H, "n_experts": E, "top_k": K, "ffn": F, "tokens": T,
                   "l2": f"weights rotate over {R} device copies, {touched / 1e6:.0f} MB touched "
                         f"per rotation vs L2 {l2 / 1e6:.0f} MB",
                   "parallelism": f"replicas x{ws}"},
        "expert_weight_gbs": gbs,
        "expert_bytes_per_step": ab["expert"], "router_bytes_per_step": ab["router"],
        "roofline": roof,
        "e2e": {"value": e2e_val, "unit": "tokens/s/layer",
                "h2d_bytes_per_step": T * H * 4, "d2h_bytes_per_step": T * H * 4},
        "gpu_launches": args.steps * q.LAUNCHES_PER_DECODE_FORWARD,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    q.qmoe_destroy(ctx)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
