"""Benchmark: qwen3moe MoE-FFN tokens/s/layer and expert-weight HBM GB/s on GB300.

Default workload (``--workload decode``): one Qwen3-30B-A3B MoE layer at decode
(hidden 2048, 128 experts, top-8 renormalised, expert FFN 768, one token, Q4_K
gate/up, Q6_K down) on seeded synthetic weights.  A step is one full MoE-FFN
layer call (router, top-k, per-expert pair lists, gate/up + SwiGLU, down,
weighted combine into the residual) through the C ABI.  Other workloads:
``batch8`` (8 tokens, Q4_K down), ``prefill`` (512 tokens, biased router, the
tensor-core path), ``step48`` (a full 48-layer decode step at context 4096) and
``prefill_layer`` (a batched prefill of 512 prompt tokens through one whole
decoder layer: attention block and MoE).

Timing: W warm-up steps, then exactly K steps replayed from CUDA graphs,
bracketed by a barrier and a device synchronise, timed with CUDA events on the
launching stream.  Every step reads a different device copy of the weights and
the copies together touch more than 4x the L2 size; right before the timed
region a buffer of twice the L2 size is written, so weight bytes come from HBM
in every timed step.  SM clocks are sampled over a window of back-to-back
replays of the same graphs around the timed region.  ``value`` is summed over
ranks (each rank runs its own replica).

``--impl reference`` times the CPU oracle (the reference arm) on the same
workload and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "qwen3moe MoE-FFN tokens/s/layer; expert-weight HBM GB/s vs GB300 peak"

WORKLOADS = {
    "decode": dict(cfg="decode", copies=32, e2e=2000, steps=20000, warmup=200,
                   desc="qwen3moe-30b-a3b MoE layer decode, T=1, Q4_K gate/up, Q6_K down"),
    "batch8": dict(cfg="batch8", copies=6, e2e=500, steps=4000, warmup=40,
                   desc="qwen3moe-30b-a3b MoE layer decode batch, T=8, Q4_K gate/up, Q4_K down"),
    "prefill": dict(cfg="prefill", copies=3, e2e=20, steps=300, warmup=6,
                    desc="qwen3moe-30b-a3b MoE layer prefill, T=512, biased router, Q6_K down"),
    "step48": dict(cfg=None, copies=1, e2e=10, steps=400, warmup=3,
                   desc="qwen3moe-30b-a3b 48-layer decode step, T=1, context 4096"),
    "prefill_layer": dict(cfg=None, copies=3, e2e=10, steps=300, warmup=6,
                          desc="qwen3moe-30b-a3b decoder layer batched prefill, T=512 prompt tokens "
                               "at positions 0..511, context 4096, Q6_K down"),
    # supplementary (not one of the five configurations): the prefill layer at
    # T=4096, where the contraction is compute-bound and the tensor-pipe
    # fraction is the meaningful one
    "prefill4096": dict(cfg="prefill", T=4096, copies=2, e2e=5, steps=60, warmup=3,
                        desc="qwen3moe-30b-a3b MoE layer prefill, T=4096, biased router, Q6_K "
                             "down (supplementary)"),
    # supplementary: the int8-activation variant (qmoe_forward_q8k) of the decode layer
    "decode_q8k": dict(cfg="decode", copies=32, e2e=2000, steps=20000, warmup=200, q8k=True,
                       desc="qwen3moe-30b-a3b MoE layer decode, T=1, Q8_K activations (int8 "
                            "variant), Q4_K gate/up, Q6_K down (supplementary)"),
    # supplementary: FP8 block-scaled experts (qmoe_forward_fp8) with the F32 router
    "decode_fp8": dict(cfg=None, fp8="decode_fp8", copies=8, e2e=2000, steps=20000, warmup=200,
                       desc="qwen3moe-30b-a3b MoE layer decode, T=1, FP8 (E4M3) experts with one "
                            "fp32 scale per 128x128 block, F32 router (supplementary)"),
    "decode_nvfp4": dict(cfg=None, nvfp4="decode_nvfp4", copies=16, e2e=2000, steps=20000,
                         warmup=200,
                         desc="qwen3moe-30b-a3b MoE layer decode, T=1, NVFP4 experts (E2M1, E4M3 "
                              "scale per 16, fp32 global per matrix), F32 router (supplementary)"),
    "prefill_nvfp4": dict(cfg=None, nvfp4="decode_nvfp4", T=512, copies=3, e2e=20, steps=300,
                          warmup=6,
                          desc="qwen3moe-30b-a3b MoE layer prefill, T=512, NVFP4 experts, F32 "
                               "router (supplementary)"),
    "prefill_fp8": dict(cfg=None, fp8="decode_fp8", T=512, copies=2, e2e=20, steps=300, warmup=6,
                        desc="qwen3moe-30b-a3b MoE layer prefill, T=512, FP8 (E4M3) experts with "
                             "one fp32 scale per 128x128 block, F32 router (supplementary)"),
}

# kernels whose summary under profiles/ carries a DRAM traffic figure
PROFILE_FOR = {"decode": "moe_decode_t1_decode_T1.md", "batch8": None, "prefill": None,
               "step48": None, "prefill4096": None, "decode_q8k": None, "prefill_layer": None,
               "decode_fp8": "moe_fp8_decode_T1.md", "prefill_fp8": None,
               "decode_nvfp4": "moe_nvfp4_decode_T1.md", "prefill_nvfp4": None}
FUSED_SOURCES = ["moe_decode_t1.cu", "kquant.cuh", "ptx_sync.cuh"]
LOWBIT_T1_SOURCES = ["moe_lowbit_t1.cu", "lowbit_items.cuh", "lowbit.cuh", "topk.cuh", "kquant.cuh", "pdl.cuh",
                     "ptx_sync.cuh"]
# the sources a profile's DRAM figure was taken on, per workload
PROFILE_SOURCES = {"decode": FUSED_SOURCES, "decode_fp8": LOWBIT_T1_SOURCES,
                   "decode_nvfp4": LOWBIT_T1_SOURCES}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS))
    ap.add_argument("--copies", type=int, default=None, help="weight copies in the rotation")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    a = ap.parse_args()
    w = WORKLOADS[a.workload]
    a.steps = w["steps"] if a.steps is None else a.steps
    a.warmup = w["warmup"] if a.warmup is None else a.warmup
    a.copies = w["copies"] if a.copies is None else a.copies
    a.e2e_steps = w["e2e"] if a.e2e_steps is None else a.e2e_steps
    return a


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            hbm = j.get("hbm_gbs") or j.get("hbm_GBps")
            tf = j.get("bf16_tflops")
            if hbm:
                return float(hbm), float(tf) if tf else FALLBACK_BF16_TFLOPS, "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def fused_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in sources or FUSED_SOURCES:
        h.update(open(os.path.join(ROOT, "quantized_mixture_experts_f32_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    name = PROFILE_FOR.get(workload)
    if not name:
        return None
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m_src = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", txt)
    if not m_src or not m_tr or m_src.group(1) != fused_source_hash(PROFILE_SOURCES.get(workload)):
        return None
    return int(m_tr.group(1))


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
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (ts, l) in self.lines if t0 <= ts <= t1] or \
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


def expert_bytes(H, F, gate_t, up_t, down_t):
    return (synth.matrix_bytes(gate_t, F, H) + synth.matrix_bytes(up_t, F, H)
            + synth.matrix_bytes(down_t, H, F))


# ----------------------------------------------------------------------------- CPU oracle

def cpu_rate(call, units: int, seconds: float, threads: int, durations=None):
    """Units per second of `call` (which processes `units`) run back to back on
    `threads` host threads for about `seconds`.  The oracle is plain C called
    through ctypes, which releases the interpreter lock for the call, and it
    keeps no global state, so the threads run it side by side.  With
    `durations` (a list), every call's own wall time in seconds is appended to
    it.  Returns (rate, calls, elapsed)."""
    counts = [0] * threads
    t0 = time.perf_counter()

    def work(i):
        while time.perf_counter() - t0 < seconds:
            c0 = time.perf_counter()
            call()
            if durations is not None:
                durations.append(time.perf_counter() - c0)
            counts[i] += 1

    ts = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    el = time.perf_counter() - t0
    return sum(counts) * units / el, sum(counts), el


def cpu_baseline(call, units: int, seconds: float, what: str):
    """The oracle on one thread and on every core: the all-core rate is the
    baseline value, the single-thread rate is kept beside it, with the median
    and the minimum of the single-thread call times (each call one repetition
    of the sample)."""
    call()
    one_calls = []
    one, n1, e1 = cpu_rate(call, units, seconds / 2, 1, one_calls)
    th = cores()
    allc, na, ea = cpu_rate(call, units, seconds / 2, th)
    return {"value": allc, "unit": "tokens/s/layer", "cores": th, "kind": "oracle",
            "single_thread_value": one,
            "single_thread_call_ms": {"median": 1e3 * float(np.median(one_calls)),
                                      "min": 1e3 * float(np.min(one_calls)),
                                      "repetitions": len(one_calls)},
            "sample": f"{what}: {n1} calls on 1 thread in {e1:.1f} s, {na} calls on {th} "
                      f"threads in {ea:.1f} s"}


def cpu_sample_layer(inp, seconds: float, max_tokens: int, q8k: bool = False):
    """The oracle on a bounded sample of the layer workload: tokens/s/layer."""
    import oracle
    oracle.build()
    forward = oracle.moe_forward_q8k if q8k else oracle.moe_forward
    n = min(inp["T"], max_tokens)
    one = dict(inp)
    one["x"] = inp["x"][:n]
    one["T"] = n
    return cpu_baseline(lambda: forward(one), n, seconds,
                        f"oracle calls on the first {n} tokens of this layer workload")


def cpu_sample_fp8(inp, seconds: float, max_tokens: int, nv: bool = False):
    """The FP8 / NVFP4 oracle on a bounded sample of the layer workload: tokens/s/layer."""
    import oracle
    oracle.build()
    n = min(inp["T"], max_tokens)
    one = dict(inp)
    one["x"] = inp["x"][:n]
    one["T"] = n
    forward = oracle.moe_forward_nvfp4 if nv else oracle.moe_forward_fp8
    return cpu_baseline(lambda: forward(one), n, seconds,
                        f"{'NVFP4' if nv else 'FP8'} oracle calls on the first {n} tokens of this "
                        "layer workload")


def cpu_sample_step(geo, seconds: float):
    import oracle
    oracle.build()
    h = synth.step_input(geo).astype(np.float64)
    pos = geo["ctx"] - 1
    small = synth.step_layer_small(geo, 0)
    ex = synth.step_layer_experts(geo, 0)
    return cpu_baseline(lambda: oracle.decode_layer(geo, small, ex, h, pos), 1, seconds,
                        "oracle decoder layers (layer 0 of the 48-layer step, context 4096)")


def cpu_sample_prefill_layer(geo, seconds: float):
    import oracle
    oracle.build()
    small = synth.step_layer_small(geo, 0)
    ex = synth.step_layer_experts(geo, 0)
    n = 4
    hs = synth.prefill_input(geo, geo["T"])[:n].astype(np.float64)
    return cpu_baseline(lambda: oracle.prefill_layer(geo, small, ex, hs, geo["pos0"]), n, seconds,
                        f"oracle layer calls on the first {n} prompt tokens (token by token)")


def cores():
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = WORKLOADS[args.workload]
    budget = 150.0
    if w.get("fp8") or w.get("nvfp4"):
        nv = bool(w.get("nvfp4"))
        inp = (synth.moe_inputs_nvfp4(synth.NVFP4_CONFIGS[w["nvfp4"]], T=w.get("T")) if nv
               else synth.moe_inputs_fp8(synth.FP8_CONFIGS[w["fp8"]], T=w.get("T")))
        sample = min(inp["T"], 8)
        one = dict(inp)
        one["x"] = inp["x"][:sample]
        one["T"] = sample
        forward = oracle.moe_forward_nvfp4 if nv else oracle.moe_forward_fp8
        step = lambda: forward(one)  # noqa: E731
        tokens_per_step = sample
        what = f"{sample} tokens of the {args.workload} layer workload per step"
    elif w["cfg"] is not None:
        inp = synth.moe_inputs(synth.MOE_CONFIGS[w["cfg"]])
        sample = min(inp["T"], 8)
        one = dict(inp)
        one["x"] = inp["x"][:sample]
        one["T"] = sample
        forward = oracle.moe_forward_q8k if w.get("q8k") else oracle.moe_forward
        step = lambda: forward(one)  # noqa: E731
        tokens_per_step = sample
        what = f"{sample} tokens of the {args.workload} layer workload per step"
    elif args.workload == "prefill_layer":
        geo = dict(synth.PREFILL_LAYER_DEFAULT)
        small = synth.step_layer_small(geo, 0)
        ex = synth.step_layer_experts(geo, 0)
        sample = 4
        hs = synth.prefill_input(geo, geo["T"])[:sample].astype(np.float64)
        step = lambda: oracle.prefill_layer(geo, small, ex, hs, geo["pos0"])  # noqa: E731
        tokens_per_step = sample
        what = f"the first {sample} prompt tokens of the prefill layer workload per step"
    else:
        geo = dict(synth.STEP_DEFAULT)
        small = synth.step_layer_small(geo, 0)
        ex = synth.step_layer_experts(geo, 0)
        h = synth.step_input(geo).astype(np.float64)
        step = lambda: oracle.decode_layer(geo, small, ex, h, geo["ctx"] - 1)  # noqa: E731
        tokens_per_step = 1
        what = "one decoder layer of the 48-layer step per step"
    t0 = time.perf_counter()
    step()
    est = time.perf_counter() - t0
    warm = min(args.warmup, 1)
    for _ in range(warm):
        step()
    # the K steps run on every host core (threads taking the next step in turn;
    # the oracle is plain C behind ctypes, which releases the interpreter lock)
    th = cores()
    k = max(3, min(args.steps, int(budget * th / max(est, 1e-6))))
    th = min(th, k)
    left = [k]
    lock = threading.Lock()

    def work():
        while True:
            with lock:
                if left[0] == 0:
                    return
                left[0] -= 1
            step()

    ts = [threading.Thread(target=work) for _ in range(th)]
    t0 = time.perf_counter()
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    el = time.perf_counter() - t0
    val = k * tokens_per_step / el
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s/layer",
            "n_gpus": args.gpus, "steps": k, "requested_steps": args.steps, "warmup": warm,
            "ms_per_step": 1000 * el / k, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w["desc"]},
            "cpu_baseline": {"value": val, "unit": "tokens/s/layer", "cores": th,
                             "kind": "oracle",
                             "sample": f"{k} steps of {what} on {th} threads (steps capped to "
                                       f"~{budget:.0f} s of single-thread work per thread)"},
            "e2e": {"value": val, "unit": "tokens/s/layer", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        pg = dist
    return ws, rank, local, pg


def timed_graphs(torch, stream, calls, steps, warmup, pg, dev, sampler_index, clock_s=1.0):
    """Capture one graph over the rotation of `calls`, replay for exactly
    `steps` steps after `warmup`; returns (ms, clocks).

    L2: right before the timed region a buffer of twice the L2 size is written,
    so no timed step finds weights that the warm-up left in L2; inside the
    region consecutive steps read different weight copies.
    Clocks: nvidia-smi samples every 100 ms, longer than a short timed region,
    so the same graphs are also replayed back to back for about `clock_s`
    seconds before and after it; the clock figures are the samples of that
    window (the timed region included)."""
    R = len(calls)
    with torch.cuda.stream(stream):
        for i in range(min(3, R)):
            calls[i]()
        stream.synchronize()
        g_full = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_full, stream=stream):
            for c in calls:
                c()
        rem = steps % R
        g_rem = None
        if rem:
            g_rem = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_rem, stream=stream):
                for c in calls[:rem]:
                    c()
        for _ in range(warmup // R):
            g_full.replay()
        for c in calls[:warmup % R]:
            c()
        stream.synchronize()
        # one full replay, timed, sizes the clock window
        t = time.perf_counter()
        g_full.replay()
        stream.synchronize()
        per_full = max(time.perf_counter() - t, 1e-6)
    n_clock = max(1, int(clock_s / 2 / per_full))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(sampler_index)
    sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        for _ in range(n_clock):
            g_full.replay()
        flush.zero_()
        if pg:
            stream.synchronize()
            pg.barrier()
        e0.record(stream)
        marks = [e0]
        for _ in range(steps // R):
            g_full.replay()
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            marks.append(ev)
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
        for _ in range(n_clock):
            g_full.replay()
    stream.synchronize()
    t1 = time.time()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    clocks = sampler.stop(t0, t1)
    clocks["window_s"] = round(t1 - t0, 3)
    ms = max_over_ranks(torch, e0.elapsed_time(e1), pg, dev)
    if clocks.get("sm_mhz"):
        clocks["ms_per_step_x_mhz"] = ms / steps * clocks["sm_mhz"]
    # the timed region in segments of one rotation each (R steps): spread of the
    # per-step time inside it
    seg = [marks[i].elapsed_time(marks[i + 1]) / R for i in range(len(marks) - 1)]
    if seg:
        clocks["segments"] = {"n": len(seg), "steps_each": R,
                              "median_ms_per_step": float(np.median(seg)),
                              "min_ms_per_step": float(np.min(seg)),
                              "max_ms_per_step": float(np.max(seg))}
    return ms, clocks


def max_over_ranks(torch, ms, pg, dev):
    """The slowest rank's time: every rank gets the same value (weak scaling
    divides the units all ranks processed by it)."""
    if not pg:
        return ms
    tt = torch.tensor([ms], dtype=torch.float64, device=dev)
    pg.all_reduce(tt, op=pg.ReduceOp.MAX)
    return float(tt.item())


def bench_layer(args, torch, q, dev, stream, ws, pg, local):
    w = WORKLOADS[args.workload]
    inp = synth.moe_inputs(synth.MOE_CONFIGS[w["cfg"]], T=w.get("T"))
    T, H, E, K, F = inp["T"], inp["H"], inp["E"], inp["K"], inp["F"]
    gt, ut, dt = q.QTYPE[inp["gate_t"]], q.QTYPE[inp["up_t"]], q.QTYPE[inp["down_t"]]
    x = torch.from_numpy(inp["x"]).to(dev)
    bias = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).to(dev)
    base = {n: torch.from_numpy(np.ascontiguousarray(inp[n])).to(dev)
            for n in ("router", "gate", "up", "down")}
    R = args.copies
    copies = [base] + [{n: t.clone() for n, t in base.items()} for _ in range(R - 1)]
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    ctx = q.qmoe_create(q.make_config(H, E, K, F, T, 1, stream.cuda_stream))
    q8k = w.get("q8k", False)
    assert not (q8k and bias is not None), "the Q8_K entry point takes no router bias"

    def mk(c):
        if q8k:
            return lambda: q.qmoe_forward_q8k(ctx, x, c["router"], c["gate"], c["up"], c["down"],
                                              gt, ut, dt, T, out)
        return lambda: q.qmoe_forward_ex(ctx, x, None, bias, c["router"], c["gate"], c["up"],
                                         c["down"], gt, ut, dt, T, out)

    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        if q8k:
            q.qmoe_forward_q8k(ctx, x, base["router"], base["gate"], base["up"], base["down"], gt,
                               ut, dt, T, out, ids, None)
        else:
            q.qmoe_forward_ex(ctx, x, None, bias, base["router"], base["gate"], base["up"],
                              base["down"], gt, ut, dt, T, out, ids, None)
    stream.synchronize()
    distinct = len(np.unique(ids.cpu().numpy()))
    ebytes = distinct * expert_bytes(H, F, inp["gate_t"], inp["up_t"], inp["down_t"])
    rbytes = E * H * 4
    ms, clocks = timed_graphs(torch, stream, [mk(c) for c in copies], args.steps, args.warmup,
                              pg, dev, local)
    secs = ms / 1e3
    step_s = secs / args.steps
    # e2e: host buffers through qmoe_forward_host (copies + sync inside every step);
    # the Q8_K entry point has no host form, so its step copies pinned x in, runs
    # the layer and copies the result out on the context's stream, then syncs
    hin = torch.from_numpy(inp["x"].copy()).pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    xin = torch.empty_like(x)

    def host_step(c):
        if q8k:
            with torch.cuda.stream(stream):
                xin.copy_(hin, non_blocking=True)
                q.qmoe_forward_q8k(ctx, xin, c["router"], c["gate"], c["up"], c["down"], gt, ut,
                                   dt, T, out)
                hout.copy_(out, non_blocking=True)
            stream.synchronize()
        else:
            q.qmoe_forward_host(ctx, hin, c["router"], c["gate"], c["up"], c["down"], gt, ut, dt,
                                T, hout)

    for i in range(3):
        host_step(copies[i % R])
    if pg:
        pg.barrier()
    te0 = time.perf_counter()
    for i in range(args.e2e_steps):
        host_step(copies[i % R])
    te = time.perf_counter() - te0
    if pg:
        tt = torch.tensor([te], device=dev)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        te = float(tt.item())
    q.qmoe_destroy(ctx)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    touched = (ebytes + rbytes) * R
    res = dict(
        value=T * args.steps * ws / secs, ms=ms, step_s=step_s, clocks=clocks,
        ebytes=ebytes, other_bytes=rbytes, distinct=distinct, T=T,
        e2e=T * args.e2e_steps * ws / te, h2d=T * H * 4, d2h=T * H * 4,
        launches=(q.LAUNCHES_PER_Q8K_FORWARD if q8k else
                  q.LAUNCHES_PER_DECODE_FORWARD if T <= 8 else q.LAUNCHES_PER_PREFILL_FORWARD),
        config={"workload": w["desc"], "hidden": H, "n_experts": E, "top_k": K, "ffn": F,
                "tokens": T, "distinct_experts": distinct,
                "l2": f"weights rotate over {R} device copies, {touched / 1e6:.0f} MB touched "
                      f"per rotation vs L2 {l2 / 1e6:.0f} MB; a {2 * l2 / 1e6:.0f} MB buffer is "
                      "written right before the timed region"},
        kernel=("whole Q8_K layer call (routing, quantise, gate/up, quantise, down, combine)"
                if q8k else "moe_decode_t1 (the whole layer is one kernel)" if T == 1
                else "moe_decode_fused (the whole layer is one kernel)" if T <= 8
                else "whole layer call (routing, gather, grouped GEMMs, combine)"))
    if q8k:
        res["dtype"] = "int8 activations (Q8_K), f32 accumulate"
    if T > 8:
        flops = T * K * 2 * (2 * F * H + H * F)
        res["tensor_tflops"] = flops / step_s / 1e12
    cpu = None
    if not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        cpu = cpu_sample_layer(inp, args.cpu_seconds, 8 if T <= 8 else 16, q8k)
    return res, cpu


def bench_layer_fp8(args, torch, q, dev, stream, ws, pg, local):
    """The MoE layer over FP8 block-scaled experts (qmoe_forward_fp8) or NVFP4
    experts (qmoe_forward_nvfp4)."""
    w = WORKLOADS[args.workload]
    nv = bool(w.get("nvfp4"))
    if nv:
        inp = synth.moe_inputs_nvfp4(synth.NVFP4_CONFIGS[w["nvfp4"]], T=w.get("T"))
        names = ("router", "gate", "gate_bs", "gate_gs", "up", "up_bs", "up_gs", "down", "down_bs",
                 "down_gs")
    else:
        inp = synth.moe_inputs_fp8(synth.FP8_CONFIGS[w["fp8"]], T=w.get("T"))
        names = ("router", "gate", "gate_scale", "up", "up_scale", "down", "down_scale")
    T, H, E, K, F = inp["T"], inp["H"], inp["E"], inp["K"], inp["F"]
    fmt = "NVFP4" if nv else "FP8"
    one = T == 1 and (H, F) == (2048, 768) and E <= 128   # the one-kernel decode
    x = torch.from_numpy(inp["x"]).to(dev)
    base = {n: torch.from_numpy(np.ascontiguousarray(inp[n])).to(dev) for n in names}
    R = args.copies
    copies = [base] + [{n: t.clone() for n, t in base.items()} for _ in range(R - 1)]
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    ctx = q.qmoe_create(q.make_config(H, E, K, F, T, 1, stream.cuda_stream))

    def fwd(c, xin, o, ids=None):
        if nv:
            q.qmoe_forward_nvfp4(ctx, xin, *[c[n] for n in names], T, o, ids, None)
        else:
            q.qmoe_forward_fp8(ctx, xin, c["router"], c["gate"], c["gate_scale"], c["up"],
                               c["up_scale"], c["down"], c["down_scale"], T, o, ids, None)

    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        fwd(base, x, out, ids)
    stream.synchronize()
    distinct = len(np.unique(ids.cpu().numpy()))
    if nv:   # codes, E4M3 block scales and the fp32 global of each matrix
        per_expert = 3 * (F * H // 2 + F * H // 16 + 4)
    else:    # codes and the fp32 block scales
        per_expert = 3 * F * H + 4 * (inp["gate_scale"][0].size + inp["up_scale"][0].size
                                      + inp["down_scale"][0].size)
    ebytes = distinct * per_expert
    rbytes = E * H * 4
    ms, clocks = timed_graphs(torch, stream, [(lambda c=c: fwd(c, x, out)) for c in copies],
                              args.steps, args.warmup, pg, dev, local)
    secs = ms / 1e3
    step_s = secs / args.steps
    # e2e: pinned host x copied in, the layer, the result copied out, then a sync
    hin = torch.from_numpy(inp["x"].copy()).pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    xin = torch.empty_like(x)

    def host_step(c):
        with torch.cuda.stream(stream):
            xin.copy_(hin, non_blocking=True)
            fwd(c, xin, out)
            hout.copy_(out, non_blocking=True)
        stream.synchronize()

    for i in range(3):
        host_step(copies[i % R])
    if pg:
        pg.barrier()
    te0 = time.perf_counter()
    for i in range(args.e2e_steps):
        host_step(copies[i % R])
    te = time.perf_counter() - te0
    if pg:
        tt = torch.tensor([te], device=dev)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        te = float(tt.item())
    q.qmoe_destroy(ctx)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    touched = (ebytes + rbytes) * R
    res = dict(
        value=T * args.steps * ws / secs, ms=ms, step_s=step_s, clocks=clocks,
        ebytes=ebytes, other_bytes=rbytes, distinct=distinct, T=T,
        e2e=T * args.e2e_steps * ws / te, h2d=T * H * 4, d2h=T * H * 4,
        launches=(q.LAUNCHES_PER_LOWBIT_T1 if one else q.LAUNCHES_PER_FP8_FORWARD if T <= 8
                  else q.LAUNCHES_PER_FP8_FORWARD + 1 if T <= q.FP8_GEMV_MAX
                  else q.LAUNCHES_PER_FP8_FORWARD_MANY),
        config={"workload": w["desc"], "hidden": H, "n_experts": E, "top_k": K, "ffn": F,
                "tokens": T, "distinct_experts": distinct, "expert_bytes": per_expert,
                "l2": f"weights rotate over {R} device copies, {touched / 1e6:.0f} MB touched "
                      f"per rotation vs L2 {l2 / 1e6:.0f} MB; a {2 * l2 / 1e6:.0f} MB buffer is "
                      "written right before the timed region"},
        kernel=(f"lowbit_t1<{fmt}> (the whole layer is one kernel)" if one
                else f"whole {fmt} layer call (router, top-k, gate/up, down, combine)"
                if T <= q.FP8_GEMV_MAX
                else f"whole {fmt} layer call (routing, gather, grouped tensor-core GEMMs, combine)"),
        dtype=(f"{'e2m1 weights and e4m3 scales' if nv else 'e4m3 weights'} widened exactly, f32 "
               "activations and accumulate" if T <= q.FP8_GEMV_MAX
               else f"{'e2m1' if nv else 'e4m3'} weights widened to f16 tensor-core operands, f32 "
                    "accumulate"))
    if T > q.FP8_GEMV_MAX:
        res["tensor_tflops"] = T * K * 2 * (2 * F * H + H * F) / step_s / 1e12
    cpu = None
    if not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        cpu = cpu_sample_fp8(inp, args.cpu_seconds, 8, nv)
    return res, cpu


def bench_step48(args, torch, q, dev, stream, ws, pg, local):
    geo = dict(synth.STEP_DEFAULT)
    L, H, E, K, F = geo["n_layers"], geo["H"], geo["E"], geo["K"], geo["F"]
    pos = geo["ctx"] - 1
    keep, structs = [], []
    ebytes = attn_bytes = kv_bytes = rbytes = 0
    for l in range(L):
        small = synth.step_layer_small(geo, l)
        ex = synth.step_layer_experts(geo, l)
        d = {}
        for n in ("attn_norm", "q_norm", "k_norm", "ffn_norm", "router", "wq", "wk", "wv", "wo"):
            d[n] = torch.from_numpy(np.ascontiguousarray(small[n])).to(dev)
        for n in ("k_cache", "v_cache"):
            d[n] = torch.from_numpy(np.ascontiguousarray(small[n]).view(np.uint16)).to(dev)
        for n in ("gate", "up", "down"):
            d[n] = torch.from_numpy(ex[n]).to(dev)
        keep.append(d)
        structs.append(q.qmoe_layer_weights(
            d["attn_norm"].data_ptr(), d["wq"].data_ptr(), d["wk"].data_ptr(), d["wv"].data_ptr(),
            d["wo"].data_ptr(), d["q_norm"].data_ptr(), d["k_norm"].data_ptr(),
            d["ffn_norm"].data_ptr(), d["router"].data_ptr(), d["gate"].data_ptr(),
            d["up"].data_ptr(), d["down"].data_ptr(), q.QTYPE[small["down_t"]],
            d["k_cache"].data_ptr(), d["v_cache"].data_ptr()))
        attn_bytes += sum(small[n].nbytes for n in ("wq", "wk", "wv", "wo"))
        kv_bytes += 2 * geo["n_kv"] * (pos + 1) * geo["head_dim"] * 2
        rbytes += small["router"].nbytes
        per = expert_bytes(H, F, "Q4_K", "Q4_K", small["down_t"])
        del ex
        keep[-1]["_per"] = per
    arr = (q.qmoe_layer_weights * L)(*structs)
    h0 = torch.from_numpy(synth.step_input(geo)).to(dev)
    hidden = torch.empty_like(h0)
    ids = torch.empty((L, K), dtype=torch.int32, device=dev)
    ctx = q.qmoe_create(q.make_config(H, E, K, F, 1, 1, stream.cuda_stream, n_heads=geo["n_heads"],
                                      n_kv_heads=geo["n_kv"], head_dim=geo["head_dim"],
                                      max_ctx=geo["ctx"], rope_base=geo["rope_base"],
                                      rms_eps=geo["eps"]))
    with torch.cuda.stream(stream):
        hidden.copy_(h0)
        q.qmoe_decode_step(ctx, arr, L, pos, hidden, ids)
    stream.synchronize()
    idn = ids.cpu().numpy()
    for l in range(L):
        ebytes += len(np.unique(idn[l])) * keep[l]["_per"]

    def step():
        hidden.copy_(h0)
        q.qmoe_decode_step(ctx, arr, L, pos, hidden)

    ms, clocks = timed_graphs(torch, stream, [step], args.steps, args.warmup, pg, dev, local)
    secs = ms / 1e3
    step_s = secs / args.steps
    hin = torch.from_numpy(synth.step_input(geo)).pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    if pg:
        pg.barrier()
    te0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        with torch.cuda.stream(stream):
            hidden.copy_(hin, non_blocking=True)
            q.qmoe_decode_step(ctx, arr, L, pos, hidden)
            hout.copy_(hidden, non_blocking=True)
        stream.synchronize()
    te = time.perf_counter() - te0
    q.qmoe_destroy(ctx)
    res = dict(
        value=L * args.steps * ws / secs, ms=ms, step_s=step_s, clocks=clocks,
        ebytes=ebytes, other_bytes=attn_bytes + kv_bytes + rbytes,
        e2e=L * args.e2e_steps * ws / te, h2d=H * 4, d2h=H * 4,
        launches=L * q.LAUNCHES_PER_DECODE_LAYER + q.LAUNCHES_PER_DECODE_STEP,
        config={"workload": WORKLOADS["step48"]["desc"], "hidden": H, "n_experts": E,
                "top_k": K, "ffn": F, "layers": L, "context": geo["ctx"], "tokens": 1,
                "l2": f"one step touches {(ebytes + attn_bytes + kv_bytes + rbytes) / 1e9:.2f} GB "
                      "vs a 136 MB L2; a buffer of twice the L2 is written right before the "
                      "timed region"},
        kernel="whole 48-layer decode step",
        tokens_per_s=args.steps * ws / secs,
        bytes_split={"experts": ebytes, "attention_weights": attn_bytes, "kv_cache": kv_bytes,
                     "routers": rbytes})
    cpu = None
    if not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        cpu = cpu_sample_step(geo, args.cpu_seconds)
    return res, cpu


def bench_prefill_layer(args, torch, q, dev, stream, ws, pg, local):
    """One whole decoder layer (attention block + MoE) over T prompt tokens
    through qmoe_prefill, the layer's weights and KV cache rotating over
    `copies` device copies."""
    geo = dict(synth.PREFILL_LAYER_DEFAULT)
    T, pos0 = geo["T"], geo["pos0"]
    H, E, K, F = geo["H"], geo["E"], geo["K"], geo["F"]
    nq, nkv, hd = geo["n_heads"], geo["n_kv"], geo["head_dim"]
    small = synth.step_layer_small(geo, 0)
    ex = synth.step_layer_experts(geo, 0)
    base = {}
    for n in ("attn_norm", "q_norm", "k_norm", "ffn_norm", "router", "wq", "wk", "wv", "wo"):
        base[n] = torch.from_numpy(np.ascontiguousarray(small[n])).to(dev)
    for n in ("k_cache", "v_cache"):
        base[n] = torch.from_numpy(np.ascontiguousarray(small[n]).view(np.uint16)).to(dev)
    for n in ("gate", "up", "down"):
        base[n] = torch.from_numpy(ex[n]).to(dev)
    R = args.copies
    copies = [base] + [{n: t.clone() for n, t in base.items()} for _ in range(R - 1)]
    dt = q.QTYPE[small["down_t"]]

    def layer_arr(d):
        return (q.qmoe_layer_weights * 1)(q.qmoe_layer_weights(
            d["attn_norm"].data_ptr(), d["wq"].data_ptr(), d["wk"].data_ptr(), d["wv"].data_ptr(),
            d["wo"].data_ptr(), d["q_norm"].data_ptr(), d["k_norm"].data_ptr(),
            d["ffn_norm"].data_ptr(), d["router"].data_ptr(), d["gate"].data_ptr(),
            d["up"].data_ptr(), d["down"].data_ptr(), dt, d["k_cache"].data_ptr(),
            d["v_cache"].data_ptr()))

    arrs = [layer_arr(c) for c in copies]
    h0 = torch.from_numpy(synth.prefill_input(geo, T)).to(dev)
    hidden = torch.empty_like(h0)
    ids = torch.empty((1, T, K), dtype=torch.int32, device=dev)
    ctx = q.qmoe_create(q.make_config(H, E, K, F, T, 1, stream.cuda_stream, n_heads=nq,
                                      n_kv_heads=nkv, head_dim=hd, max_ctx=geo["ctx"],
                                      rope_base=geo["rope_base"], rms_eps=geo["eps"]))
    with torch.cuda.stream(stream):
        hidden.copy_(h0)
        q.qmoe_prefill(ctx, arrs[0], 1, T, pos0, hidden, ids)
    stream.synchronize()
    distinct = len(np.unique(ids.cpu().numpy()))
    ebytes = distinct * expert_bytes(H, F, "Q4_K", "Q4_K", small["down_t"])
    attn_bytes = sum(small[n].nbytes for n in ("wq", "wk", "wv", "wo"))
    qd, kvd = nq * hd, nkv * hd
    keys = sum(pos0 + t + 1 for t in range(T))
    # KV: the batch's slots written once, every visible key row read once per kv head
    kv_bytes = 2 * 2 * T * kvd + 2 * 2 * nkv * hd * (pos0 + T)
    rbytes = small["router"].nbytes
    flops = (T * K * 2 * (2 * F * H + H * F) + 2 * T * (qd + 2 * kvd) * H + 2 * T * H * qd
             + 4 * nq * hd * keys)

    def mk(a):
        def step():
            hidden.copy_(h0)
            q.qmoe_prefill(ctx, a, 1, T, pos0, hidden)
        return step

    ms, clocks = timed_graphs(torch, stream, [mk(a) for a in arrs], args.steps, args.warmup,
                              pg, dev, local)
    secs = ms / 1e3
    step_s = secs / args.steps
    hin = torch.from_numpy(synth.prefill_input(geo, T)).pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    for i in range(2):
        with torch.cuda.stream(stream):
            hidden.copy_(hin, non_blocking=True)
            q.qmoe_prefill(ctx, arrs[i % R], 1, T, pos0, hidden)
            hout.copy_(hidden, non_blocking=True)
        stream.synchronize()
    if pg:
        pg.barrier()
    te0 = time.perf_counter()
    for i in range(args.e2e_steps):
        with torch.cuda.stream(stream):
            hidden.copy_(hin, non_blocking=True)
            q.qmoe_prefill(ctx, arrs[i % R], 1, T, pos0, hidden)
            hout.copy_(hidden, non_blocking=True)
        stream.synchronize()
    te = time.perf_counter() - te0
    if pg:
        tt = torch.tensor([te], device=dev)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        te = float(tt.item())
    q.qmoe_destroy(ctx)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    touched = (ebytes + attn_bytes + rbytes) * R
    res = dict(
        value=T * args.steps * ws / secs, ms=ms, step_s=step_s, clocks=clocks,
        ebytes=ebytes, other_bytes=attn_bytes + kv_bytes + rbytes, distinct=distinct, T=T,
        e2e=T * args.e2e_steps * ws / te, h2d=T * H * 4, d2h=T * H * 4,
        launches=q.LAUNCHES_PER_PREFILL_LAYER_ATTN + q.LAUNCHES_PER_PREFILL_FORWARD,
        tensor_tflops=flops / step_s / 1e12,
        config={"workload": WORKLOADS["prefill_layer"]["desc"], "hidden": H, "n_experts": E,
                "top_k": K, "ffn": F, "n_heads": nq, "n_kv_heads": nkv, "head_dim": hd,
                "tokens": T, "pos0": pos0, "context": geo["ctx"], "distinct_experts": distinct,
                "l2": f"weights rotate over {R} device copies, {touched / 1e6:.0f} MB touched "
                      f"per rotation vs L2 {l2 / 1e6:.0f} MB; a {2 * l2 / 1e6:.0f} MB buffer is "
                      "written right before the timed region"},
        kernel="whole layer call (attention block GEMMs and attention, routing, grouped GEMMs, "
               "combine)",
        tokens_per_s=T * args.steps * ws / secs,
        bytes_split={"experts": ebytes, "attention_weights": attn_bytes, "kv_cache": kv_bytes,
                     "routers": rbytes},
        flops_per_step=flops)
    cpu = None
    if not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        cpu = cpu_sample_prefill_layer(geo, args.cpu_seconds)
    return res, cpu


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    ws, rank, local, pg = dist_init()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    try:
        # device memory in use before this run allocates anything: its own CUDA
        # context plus whatever other processes hold on the GPU
        free0, total0 = torch.cuda.mem_get_info(dev)
        gpu_mem = {"total_mib": total0 >> 20, "used_before_run_mib": (total0 - free0) >> 20}
    except Exception as e:  # recorded, never fatal
        gpu_mem = {"error": str(e)}
    import quantized_mixture_experts_f32_gb300 as q
    stream = torch.cuda.Stream(dev)
    if args.workload == "step48":
        res, cpu = bench_step48(args, torch, q, dev, stream, ws, pg, local)
    elif args.workload == "prefill_layer":
        res, cpu = bench_prefill_layer(args, torch, q, dev, stream, ws, pg, local)
    elif WORKLOADS[args.workload].get("fp8") or WORKLOADS[args.workload].get("nvfp4"):
        res, cpu = bench_layer_fp8(args, torch, q, dev, stream, ws, pg, local)
    else:
        res, cpu = bench_layer(args, torch, q, dev, stream, ws, pg, local)
    hbm, tf, kind = peaks()
    step_s = res["step_s"]
    gbs = res["ebytes"] / step_s / 1e9
    all_gbs = (res["ebytes"] + res["other_bytes"]) / step_s / 1e9
    traffic = profiled_traffic(args.workload)
    roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
            "peak_kind": kind, "traffic": traffic, "kernel": res["kernel"],
            "algorithmic_bytes_per_launch": res["ebytes"],
            "achieved_all_bytes": all_gbs, "frac_all_bytes": all_gbs / hbm,
            "frac_of_nominal_8tbs": gbs / 8000.0}
    line = {
        "metric": METRIC, "value": res["value"], "unit": "tokens/s/layer", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict(res["config"], parallelism=f"replicas x{ws}"),
        "expert_weight_gbs": gbs, "roofline": roof,
        "e2e": {"value": res["e2e"], "unit": "tokens/s/layer", "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"]},
        "gpu_launches": args.steps * res["launches"],
        "clocks": res["clocks"],
        "gpu_memory": gpu_mem,
    }
    if "dtype" in res:
        line["dtype"] = res["dtype"]
    if "tensor_tflops" in res:
        line["dtype"] = "f16 tensor-core operands, f32 accumulate"
        line["tensor"] = {"achieved_tflops": res["tensor_tflops"], "peak_tflops": tf,
                          "frac": res["tensor_tflops"] / tf, "peak_kind": kind}
        if "flops_per_step" in res:
            line["tensor"]["flops_per_step"] = res["flops_per_step"]
    if "bytes_split" in res:
        line["tokens_per_s"] = res["tokens_per_s"]
        line["bytes_per_step"] = res["bytes_split"]
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
