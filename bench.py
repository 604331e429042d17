#!/usr/bin/env python
"""Prefill-GEMM benchmark of one Qwen2.5-7B-shaped layer on GB300.

One step = the layer's seven prefill GEMMs Y = X . W^T at M = 2048 tokens
through the library's public calls: mq_gemm_grouped for the projections
that share their input (q|k|v, gate|up: one launch each) and mq_gemm_auto
for o and down (the M gate sends M = 2048 to the cached path).  All are the
tcgen05 GEMM on the f16 cache, with a split-K tail + fixed-order reduce
where a tile grid's last wave underfills the GPU.  Weights q/k/v/o/gate/up are
Q4_K, down is Q6_K, all seeded synthetic bytes with the model's shapes; they
are registered (decoded once into the f16 cache) before timing.

Printed: one JSON line (rank 0) with the contract keys plus
  roofline      the cached GEMM kernel against the measured dense peak, its
                per-launch duration read from CUDA events that the library
                records on the launching stream during the timed steps;
  cpu_baseline  the CPU oracle (f64) on a bounded sample of the same layer;
  e2e           the same metric with host buffers: pinned-host inputs copied
                in and all outputs copied out inside the timed region;
  decode        the one-time decoders (registration, cold) against HBM bandwidth;
  decode_steady the decoders back to back on the 7B gate/down shapes and
                weights of the other formats at the gate's shape (HBM GB/s);
  small_m       fused vs cached over the small-M sweep, back to back over
                rotating weight copies (crossover, HBM GB/s);
  more_formats  Q4_0 / Q5_0 / Q5_1 / Q5_K at the 7B gate and down shapes:
                fused and cached at M = 32 and 2048, same method;
  triangle      the 7B layer's seven GEMMs one call each through the cached
                path, the per-call scratch mode and the fused path at M = 32
                and 2048 (and the fused path grouped as q|k|v, o, gate|up,
                down): time per layer and device bytes each mode holds;
  row_pad       F16 / BF16 weights of the Llama-3.1-8B layer's shapes at
                M = 512, cached GEMM on the row-padded copy vs unpadded rows;
  e4m3          the same layer step through the 8-bit variant (its own
                numeric contract): the four distinct activations quantized
                per step, seven e4m3 GEMMs; TFLOP/s, the e4m3 kernel against
                the 8-bit dense peak, distance to the f16 result.

--impl reference times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from quantized_weight_prefill_gguf_gb300 import synth  # noqa: E402

METRIC = "prefill GEMM TFLOP/s & tok/s per 7B layer at M=2048; % of f16 TC / HBM roofline"
WORKLOAD = "qwen2.5-7b_layer"
M_TOKENS = 2048
L2_BYTES = 126 * 1024 * 1024


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def cached_kernel_source_hash() -> str:
    """sha256 over the sources that make up the cached GEMM kernel."""
    h = hashlib.sha256()
    for f in ("gemm.cu", "mq_tile.cuh", "mq_ptx.cuh", "mq_internal.h", "mq_launch.cuh"):
        with open(os.path.join(ROOT, "quantized_weight_prefill_gguf_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def layer_flops(weights, M):
    return sum(2.0 * M * w.N * w.K for w in weights)


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, ms_per_step: float) -> float:
    """Weak scaling: every rank runs its own step, the job does world steps
    in the slowest rank's time."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_path: str | None = None):
        self.gpu = gpu_index
        self.out_path = out_path
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if self.out_path:
            with open(self.out_path, "w") as fh:
                fh.write("\n".join(self.lines) + "\n")
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- reference arm (CPU oracle)

def oracle_cpu_run(weights, xs, budget_s: float, min_tokens: int = 1):
    """Time the oracle's f64 GEMM over the layer on a token sample sized to
    about budget_s seconds.  Returns (tflops, tokens, seconds, decode_s, threads)."""
    import oracle
    orc = oracle.load()
    t0 = time.perf_counter()
    W16 = [orc.decode_matrix(w.qtype, w.data, w.N, w.K) for w in weights]
    decode_s = time.perf_counter() - t0
    # calibrate on 4 tokens, then size the sample
    t0 = time.perf_counter()
    for w, W in zip(weights, W16):
        orc.gemm_f64(xs[w.K][:4].view(np.uint16), W)
    cal = time.perf_counter() - t0
    per_token = cal / 4
    tokens = int(max(min_tokens, min(M_TOKENS, budget_s / max(per_token, 1e-9))))
    t0 = time.perf_counter()
    for w, W in zip(weights, W16):
        orc.gemm_f64(xs[w.K][:tokens].view(np.uint16), W)
    secs = time.perf_counter() - t0
    tflops = layer_flops(weights, tokens) / secs / 1e12
    return tflops, tokens, secs, decode_s, orc.num_threads()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    weights, xs = synth.workload(WORKLOAD, seed=0)
    import oracle
    orc = oracle.load()
    W16 = [orc.decode_matrix(w.qtype, w.data, w.N, w.K) for w in weights]
    # size each step so the whole run takes about two minutes
    t0 = time.perf_counter()
    for w, W in zip(weights, W16):
        orc.gemm_f64(xs[w.K][:2].view(np.uint16), W)
    per_token = (time.perf_counter() - t0) / 2
    budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(max(1, min(M_TOKENS, budget / per_token)))

    def step():
        for w, W in zip(weights, W16):
            orc.gemm_f64(xs[w.K][:tokens].view(np.uint16), W)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    flops = layer_flops(weights, tokens) * args.steps
    value = flops / secs / 1e12
    sample = (f"{tokens} of the {M_TOKENS} tokens per step through all 7 GEMMs of the layer "
              f"(f64 accumulation, weights decoded once by the oracle before timing)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_TOKENS, "tokens_per_step_sampled": tokens},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- our arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle sample budget for cpu_baseline")
    ap.add_argument("--no-extras", action="store_true", help="skip e2e, small-M sweep and cpu_baseline")
    ap.add_argument("--clocks-out", default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import quantized_weight_prefill_gguf_gb300 as mq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()

    P = peaks()
    weights, xs = synth.workload(WORKLOAD, seed=0)
    # each rank processes its own batch of tokens (independent prefill u-batches)
    if rank > 0:
        g = synth.rng(1000 + rank)
        xs = {k: synth.activations(g, M_TOKENS, k) for k in xs}

    stream = torch.cuda.current_stream()
    qdev = [torch.from_numpy(w.data).cuda() for w in weights]
    torch.cuda.synchronize()

    # registration = one-time decode into the f16 caches, traced per weight
    mq.mq_trace_enable(True)
    handles = [mq.mq_register_weight(w.qtype, q, w.N, w.K) for w, q in zip(weights, qdev)]
    torch.cuda.synchronize()
    dec = [r for r in mq.mq_trace_records() if r["kind"] == mq.MQ_TRACE_DECODE]
    mq.mq_trace_enable(False)
    decode_bytes = sum(synth.nblocks(w.qtype, w.N, w.K) * synth.BLOCK[w.qtype][1] + 2 * w.N * w.K for w in weights)
    decode_ms = sum(r["ms_main"] for r in dec)

    xdev = {k: torch.from_numpy(v).cuda() for k, v in xs.items()}
    ys = [torch.empty((M_TOKENS, w.N), dtype=torch.float32, device="cuda") for w in weights]
    mq.mq_reserve_workspace(64 << 20)

    def step(xmap):
        layer_step(mq, weights, handles, ys, xmap, M_TOKENS, stream)

    for _ in range(args.warmup):
        step(xdev)
    torch.cuda.synchronize()
    mq.mq_stream_status()

    # ---- timed region
    clocks = ClockSampler(local_rank, args.clocks_out)
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = mq.mq_launch_count()
    barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        step(xdev)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    launches = mq.mq_launch_count() - launches0
    clk = clocks.stop()
    mq.mq_stream_status()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist, "cuda")

    # Per-kernel durations for the roofline: a separate pass with the
    # library's trace events (events recorded between two launches end the
    # overlap that programmatic dependent launch gives, so the timed steps
    # above run without them).
    trace_steps = min(args.steps, 200)
    mq.mq_trace_enable(True)
    for _ in range(trace_steps):
        step(xdev)
    torch.cuda.synchronize()
    mq.mq_trace_enable(False)

    flops_step = layer_flops(weights, M_TOKENS)
    value = whole_job_tflops(world, flops_step, ms)

    # ---- roofline of the dominant kernel: the cached GEMM (k_gemm_cached)
    recs = mq.mq_trace_records()
    gem = [r for r in recs if r["kind"] == mq.MQ_TRACE_GEMM_CACHED]
    g_flops = sum(2.0 * r["M"] * r["N"] * r["K"] for r in gem)
    g_ms = sum(r["ms_main"] for r in gem)
    red_ms = sum(r["ms_aux"] for r in gem)
    per_gemm = []
    for grp in LAUNCH_GROUPS:
        ws_ = [w for w in weights if w.name in grp]
        n_tot, K_ = sum(w.N for w in ws_), ws_[0].K
        rs = [r for r in gem if r["N"] == n_tot and r["K"] == K_]
        if rs:
            t_main = statistics.median(r["ms_main"] for r in rs)
            t_aux = statistics.median(r["ms_aux"] for r in rs)
            per_gemm.append({"name": "|".join(grp), "N": n_tot, "K": K_,
                             "type": "/".join(sorted({synth.TYPE_NAME[w.qtype] for w in ws_})),
                             "gemm_us": t_main * 1e3, "reduce_us": t_aux * 1e3,
                             "tflops": 2.0 * M_TOKENS * n_tot * K_ / ((t_main + t_aux) * 1e-3) / 1e12})
    n_launch = max(1, len(gem))
    achieved = (g_flops / n_launch) / ((g_ms / n_launch) * 1e-3) / 1e12 if g_ms > 0 else None
    traffic = None
    tp = os.path.join(ROOT, "profiles", "k_gemm_cached.qwen2.5-7b_layer.traffic.json")
    if os.path.exists(tp):
        with open(tp) as fh:
            rec = json.load(fh)
        # the counters only describe the kernel source they were taken from
        if rec.get("kernel_source_sha256") == cached_kernel_source_hash():
            traffic = rec.get("k_gemm_cached_bytes_per_launch")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": P["bf16_tflops"], "unit": "TFLOP/s",
                "frac": (achieved / P["bf16_tflops"]) if achieved else None, "traffic": traffic,
                "kernel": "k_gemm_cached (tcgen05 f16 GEMM on the f16 cache)",
                "peak_kind": f"dense bf16 burst ({P['source']}); f16 nominal rate equals bf16",
                "frac_of_sustained": (achieved / P["bf16_tflops_sustained"]) if achieved else None,
                "launches_traced": len(gem), "traced_steps": trace_steps,
                "reduce_ms_per_step": red_ms / trace_steps}

    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_TOKENS, "gemms": [w.name for w in weights],
                   "weights": "q/k/v/o/gate/up Q4_K, down Q6_K (seeded synthetic blocks, model shapes)",
                   "gflop_per_step": flops_step / 1e9,
                   "path": "mq_gemm_grouped (q|k|v, gate|up) + mq_gemm_auto -> cached (o, down)",
                   "l2": "inputs larger than L2: 466 MB of f16 weight caches per step vs 126 MB L2",
                   "parallelism": f"replicas x{world} (independent token batches)"},
        "tok_per_s_per_layer": world * M_TOKENS / (ms * 1e-3),
        "tok_per_s_28_layer_gemms_only": world * M_TOKENS / (28 * ms * 1e-3),
        "frac_of_peak": value / world / P["bf16_tflops"],
        "roofline": roofline,
        "per_gemm": per_gemm,
        "gpu_launches": launches,
        "clocks": clk,
        "decode": {"bytes": decode_bytes, "ms": decode_ms,
                   "gbs": decode_bytes / (decode_ms * 1e-3) / 1e9 if decode_ms else None,
                   "frac_hbm": (decode_bytes / (decode_ms * 1e-3) / 1e9) / P["hbm_gbs"] if decode_ms else None,
                   "note": "one-time registration decode of the 7 weights (blocks read + f16 written), cold"},
    }

    if not args.no_extras:
        out["e2e"] = e2e_run(mq, torch, weights, handles, xs, ys, stream, min(args.steps, 50), flops_step, dist)
        out["small_m"] = small_m_sweep(mq, torch, stream, P)
        out["decode_steady"] = decode_steady(mq, torch, stream, P)
        out["more_formats"] = more_formats(mq, torch, stream, P)
        out["triangle"] = triangle(mq, torch, stream, weights, handles, qdev, xdev)
        out["row_pad"] = row_pad(mq, torch, stream)
        out["e4m3"] = e4m3_layer(mq, torch, stream, weights, qdev, xdev, ys, P, min(args.steps, 400), flops_step)
    if rank == 0 and world == 1 and not args.no_extras:
        tf, tokens, secs, dsec, threads = oracle_cpu_run(weights, xs, args.cpu_seconds)
        out["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                               "sample": f"{tokens} of {M_TOKENS} tokens through all 7 GEMMs (f64, {secs:.1f} s); "
                                         f"oracle decode of the 7 weights took {dsec:.1f} s before"}
    for h in handles:
        h.release()
    if rank == 0:
        print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()
    return 0


# The layer's GEMMs as launched: the projections that read the same
# activations go out as one grouped launch (q|k|v on the attention input,
# gate|up on the MLP input); o and down take the M gate (mq_gemm_auto).
LAUNCH_GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def layer_step(mq, weights, handles, ys, xmap, M, stream):
    by_name = {w.name: i for i, w in enumerate(weights)}
    for grp in LAUNCH_GROUPS:
        idx = [by_name[n] for n in grp]
        x = xmap[weights[idx[0]].K]
        if len(idx) == 1:
            mq.mq_gemm_auto(x, handles[idx[0]], ys[idx[0]], M, stream)
        else:
            mq.mq_gemm_grouped(x, [handles[i] for i in idx], [ys[i] for i in idx], M, stream)


def e2e_run(mq, torch, weights, handles, xs, ys, stream, steps, flops_step, dist):
    """The step through the public API with host buffers: every step copies
    its activations in from pinned host memory and all seven outputs back to
    pinned host memory, inside the timed region.  Copies run on their own
    streams with two sets of device buffers, as a serving loop would: step
    t's outputs go out while step t+1's inputs come in and its GEMMs run."""
    xh = {k: torch.from_numpy(v).pin_memory() for k, v in xs.items()}
    xd = [{k: torch.empty(v.shape, dtype=torch.float16, device="cuda") for k, v in xs.items()} for _ in range(2)]
    yd = [ys, [torch.empty_like(y) for y in ys]]
    yh = [[torch.empty(y.shape, dtype=torch.float32).pin_memory() for y in ys] for _ in range(2)]
    h2d = sum(v.numel() * 2 for v in xh.values())
    d2h = sum(y.numel() * 4 for y in ys)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done = [ev(), ev()]
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    used = [False, False]

    def step(t):
        b = t & 1
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(comp_done[b])          # x buffer b free again
            for k in xh:
                xd[b][k].copy_(xh[k], non_blocking=True)
            in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if used[b]:
            stream.wait_event(out_done[b])             # y buffers b copied out
        layer_step(mq, weights, handles, yd[b], xd[b], M_TOKENS, stream)
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for y, yhost in zip(yd[b], yh[b]):
                yhost.copy_(y, non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    for t in range(4):
        step(t)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for t in range(steps):
        step(t)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, dist, "cuda")
    world = dist.get_world_size() if dist is not None else 1
    return {"value": whole_job_tflops(world, flops_step, ms), "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "copies": "pinned host <-> device on two copy streams, double-buffered device X and Y"}


def _rotating_time_us(torch, fns, stream, reps=5):
    """Median per-call device time of the calls in `fns`, issued back to back
    on `stream` (CUDA events around the whole run of calls)."""
    for fn in fns:
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for fn in fns:
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3 / len(fns))
    return statistics.median(ts)


def _fused_vs_cached(mq, torch, stream, P, w, x_all, ms):
    """Rows {name, M, copies, <path>_us/_tflops/_gbs/_frac_hbm} for weight w
    at each M: per-call time of calls issued back to back over R registered
    copies of the weight, R chosen so the weights touched (raw blocks for
    fused, f16 caches for cached) exceed 400 MB, three times the L2: every
    call streams its weight from HBM, as in a layer stack, and the launch gap
    between calls is included."""
    raw_bytes = synth.nblocks(w.qtype, w.N, w.K) * synth.BLOCK[w.qtype][1]
    R = max(3, -(-(400 << 20) // raw_bytes))
    qs = [torch.from_numpy(w.data).cuda() for _ in range(R)]
    hs = [mq.mq_register_weight(w.qtype, q, w.N, w.K) for q in qs]
    rows = []
    for M in ms:
        x = x_all[:M].contiguous()
        y = torch.empty((M, w.N), dtype=torch.float32, device="cuda")
        row = {"name": w.name, "M": M, "copies": R}
        for path, fn in (("fused", mq.mq_gemm_fused), ("cached", mq.mq_gemm)):
            calls = [functools.partial(fn, x, h, y, M, stream) for h in hs]
            t_us = _rotating_time_us(torch, calls, stream)
            wbytes = raw_bytes if path == "fused" else 2 * w.N * w.K
            byts = wbytes + 2 * M * w.K + 4 * M * w.N
            row[path + "_us"] = t_us
            row[path + "_tflops"] = 2.0 * M * w.N * w.K / (t_us * 1e-6) / 1e12
            row[path + "_gbs"] = byts / (t_us * 1e-6) / 1e9
            row[path + "_frac_hbm"] = row[path + "_gbs"] / P["hbm_gbs"]
        rows.append(row)
    mq.mq_stream_status()
    for h in hs:
        h.release()
    del qs
    return rows


def small_m_sweep(mq, torch, stream, P):
    """Fused vs cached on the 7B gate (Q4_K 18944x3584) and down (Q6_K
    3584x18944) shapes over the M sweep (rotating weight copies)."""
    weights, xs = synth.workload("small_m_sweep", seed=0)
    res = []
    for w in weights:
        if w.name == "up":
            continue
        x_all = torch.from_numpy(xs[w.K]).cuda()
        res += _fused_vs_cached(mq, torch, stream, P, w, x_all, synth.WORKLOADS["small_m_sweep"][1])
    cross = {}
    for name in ("gate", "down"):
        ms_ = [r["M"] for r in res if r["name"] == name and r["cached_us"] <= r["fused_us"]]
        cross[name] = min(ms_) if ms_ else None
    return {"rows": res, "cached_wins_from_M": cross, "gate_in_use": mq.mq_get_m_gate(),
            "method": "back to back over rotating weight copies (> 3x L2), per-call average including launch gaps"}


def more_formats(mq, torch, stream, P):
    """Q4_0 / Q5_0 / Q5_1 / Q5_K weights at the 7B gate (18944x3584) and down
    (3584x18944) shapes, fused and cached at M = 32 and 2048 (rotating
    weight copies, as for the small-M sweep)."""
    weights, xs = synth.workload("more_formats", seed=0)
    res = []
    for w in weights:
        x_all = torch.from_numpy(xs[w.K]).cuda()
        res += _fused_vs_cached(mq, torch, stream, P, w, x_all, synth.WORKLOADS["more_formats"][1])
    return {"rows": res, "method": "back to back over rotating weight copies (> 3x L2), per-call average"}


def triangle(mq, torch, stream, weights, handles, qdev, xs):
    """The pages' time-vs-memory triangle on the 7B layer: each of the seven
    GEMMs as its own call (no grouping) through the cached path (resident
    f16 caches), the per-call scratch mode (one f16 scratch as large as the
    largest weight, re-decoded every call) and the fused path (raw blocks
    only), and the fused path once more in the layer's four launch groups
    (q|k|v and gate|up as one mq_gemm_fused_grouped call each).  Time per
    layer = the calls back to back, median of 5."""
    fused_h = [mq.mq_register_weight(w.qtype, q, w.N, w.K, flags=mq.MQ_REG_NO_CACHE)
               for w, q in zip(weights, qdev)]
    scratch_elems = max(w.N * h.info()[2] for w, h in zip(weights, handles))
    scratch = torch.empty(scratch_elems, dtype=torch.float16, device="cuda")
    cache_bytes = sum(2 * w.N * h.info()[2] for w, h in zip(weights, handles))
    raw_bytes = sum(w.data.size for w in weights)
    rows = []
    for M in (32, 2048):
        ys = [torch.empty((M, w.N), dtype=torch.float32, device="cuda") for w in weights]
        xm = {K: x[:M].contiguous() for K, x in xs.items()}
        modes = {
            "cached": [functools.partial(mq.mq_gemm, xm[w.K], h, y, M, stream)
                       for w, h, y in zip(weights, handles, ys)],
            "scratch": [functools.partial(mq.mq_gemm_scratch, xm[w.K], h, y, scratch, M, stream)
                        for w, h, y in zip(weights, handles, ys)],
            "fused": [functools.partial(mq.mq_gemm_fused, xm[w.K], h, y, M, stream)
                      for w, h, y in zip(weights, fused_h, ys)],
            "fused_grouped": [functools.partial(mq.mq_gemm_fused_grouped, xm[weights[idx[0]].K],
                                                [fused_h[i] for i in idx], [ys[i] for i in idx], M, stream)
                              for idx in ([i for i, w in enumerate(weights) if w.name in grp] for grp in LAUNCH_GROUPS)],
        }
        row = {"M": M}
        for name, calls in modes.items():
            row[name + "_us_per_layer"] = _rotating_time_us(torch, calls, stream) * len(calls)
        rows.append(row)
    mq.mq_stream_status()
    for h in fused_h:
        h.release()
    return {"rows": rows, "device_bytes": {"cached": raw_bytes + cache_bytes,
                                           "scratch": raw_bytes + 2 * scratch_elems, "fused": raw_bytes},
            "method": "seven single calls back to back (layer weights 148 MB raw / 466 MB f16, > L2); "
                      "fused_grouped: four calls (q|k|v and gate|up through mq_gemm_fused_grouped)"}


def row_pad(mq, torch, stream):
    """Cached GEMM at M = 512 on F16 / BF16 weights of the Llama-3.1-8B
    layer's shapes, rows padded by 128 bytes (the default for K = 4096 and
    14336) vs unpadded (MQ_REG_NO_KPAD), back to back over R registered
    copies (> 400 MB of weights touched)."""
    weights, xs = synth.workload("float_layer", seed=0)
    M = 512
    res = []
    for w in weights:
        x = torch.from_numpy(xs[w.K][:M]).cuda()
        y = torch.empty((M, w.N), dtype=torch.float32, device="cuda")
        R = max(3, -(-(400 << 20) // (2 * w.N * w.K)))
        qs = [torch.from_numpy(w.data).cuda() for _ in range(R)]
        row = {"name": w.name, "M": M, "copies": R}
        for label, flags in (("padded", 0), ("unpadded", mq.MQ_REG_NO_KPAD)):
            hs = [mq.mq_register_weight(w.qtype, q, w.N, w.K, flags=flags) for q in qs]
            t_us = _rotating_time_us(torch, [functools.partial(mq.mq_gemm, x, h, y, M, stream) for h in hs], stream)
            row[label + "_us"] = t_us
            row[label + "_tflops"] = 2.0 * M * w.N * w.K / (t_us * 1e-6) / 1e12
            row[label + "_ldk"] = hs[0].info()[2]
            for h in hs:
                h.release()
        res.append(row)
        del qs
    mq.mq_stream_status()
    return {"rows": res, "method": "back to back over R registered copies, each from its own weight buffer "
                                   "(an unpadded F16 weight is read in place)"}


def e4m3_layer(mq, torch, stream, weights, qdev, xdev, ys_f16, P, steps, flops_step):
    """The layer step on the 8-bit variant: per step the activations of the
    four launch groups (q|k|v, o, gate|up, down) are quantized once each and
    the seven GEMMs run on e4m3 operands, grouped as in the f16 step.  Timed like the main loop (CUDA
    events around `steps` steps after 5 warm-ups); the e4m3 kernel's mean
    launch time comes from a traced pass."""
    M = M_TOKENS
    hs = [mq.mq_register_weight(w.qtype, q, w.N, w.K, flags=mq.MQ_REG_E4M3) for w, q in zip(weights, qdev)]
    groups = [g for g in LAUNCH_GROUPS]
    idx = {w.name: i for i, w in enumerate(weights)}
    x8 = {}
    for g in groups:
        K = weights[idx[g[0]]].K
        x8[g] = (torch.empty((M, K), dtype=torch.uint8, device="cuda"), torch.empty(M, dtype=torch.float32,
                                                                                     device="cuda"))
    ys = [torch.empty((M, w.N), dtype=torch.float32, device="cuda") for w in weights]

    def step():
        for g in groups:
            K = weights[idx[g[0]]].K
            q8, sx = x8[g]
            mq.mq_quantize_e4m3(xdev[K][:M], q8, sx, stream)
            members = [idx[name] for name in g]
            if len(members) == 1:
                mq.mq_gemm_e4m3(q8, sx, hs[members[0]], ys[members[0]], M, stream)
            else:
                mq.mq_gemm_e4m3_grouped(q8, sx, [hs[i] for i in members], [ys[i] for i in members], M, stream)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    mq.mq_trace_enable(True)
    for _ in range(20):
        step()
    torch.cuda.synchronize()
    recs = [r for r in mq.mq_trace_records() if r["kind"] == mq.MQ_TRACE_GEMM_CACHED]
    mq.mq_trace_enable(False)
    kern_flops = [2.0 * r["M"] * r["N"] * r["K"] for r in recs]
    kern_ms = [r["ms_main"] for r in recs]
    achieved = sum(kern_flops) / (sum(kern_ms) * 1e-3) / 1e12 if recs else None
    peak8 = 2.0 * P["bf16_tflops"]
    gi = idx["gate"]
    dist = float(torch.linalg.norm(ys[gi] - ys_f16[gi]) / torch.linalg.norm(ys_f16[gi]))
    mq.mq_stream_status()
    for h in hs:
        h.release()
    small = _e4m3_small_m(mq, torch, stream, weights[gi], qdev[gi], xdev, P)
    return {"ms_per_step": ms, "tflops": flops_step / (ms * 1e-3) / 1e12, "steps": steps, "small_m": small,
            "kernel": {"name": "k_gemm_e4m3", "achieved_tflops": achieved, "peak_tflops": peak8,
                       "peak_note": "8-bit dense = 2 x the measured bf16 burst peak (the nominal fp8:bf16 ratio)",
                       "frac": achieved / peak8 if achieved else None},
            "rel_distance_to_f16_gate": dist,
            "note": "separate numeric contract: e4m3 operands with per-row / per-token f32 scales"}


def _e4m3_small_m(mq, torch, stream, w, q, xdev, P):
    """The e4m3 GEMM on the 7B gate shape at small M, where it streams one
    byte per weight: back to back over R registered copies (> 400 MB of e4m3
    weights touched), activations quantized once per M."""
    wbytes = w.N * w.K + 4 * w.N
    R = max(3, -(-(400 << 20) // wbytes))
    qs = [q.clone() for _ in range(R)]
    hs = [mq.mq_register_weight(w.qtype, qq, w.N, w.K, flags=mq.MQ_REG_E4M3) for qq in qs]
    rows = []
    for M in (1, 32, 128):
        x8 = torch.empty((M, w.K), dtype=torch.uint8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        mq.mq_quantize_e4m3(xdev[w.K][:M], x8, sx, stream)
        y = torch.empty((M, w.N), dtype=torch.float32, device="cuda")
        t_us = _rotating_time_us(torch, [functools.partial(mq.mq_gemm_e4m3, x8, sx, h, y, M, stream) for h in hs],
                                 stream)
        byts = wbytes + M * w.K + 4 * M + 4 * M * w.N
        rows.append({"M": M, "us": t_us, "gbs": byts / (t_us * 1e-6) / 1e9,
                     "frac_hbm": byts / (t_us * 1e-6) / 1e9 / P["hbm_gbs"]})
    mq.mq_stream_status()
    for h in hs:
        h.release()
    del qs
    return {"weight": f"{w.name} {w.N}x{w.K}", "copies": R, "rows": rows}


def decode_steady(mq, torch, stream, P):
    """Standalone decoders (mq_dequantize) on the 7B gate (Q4_K), down (Q6_K)
    and 18944x3584 weights of the other formats: per-call time of back-to-back calls over
    three input copies into one f16 output (output 136 MB, larger than L2)."""
    g = synth.rng(7)
    out = {}
    shapes = [(synth.Q4_K, 18944, 3584), (synth.Q6_K, 3584, 18944)]
    shapes += [(qt, 18944, 3584) for qt in (synth.Q8_0, synth.Q4_0, synth.Q5_0, synth.Q5_1, synth.Q5_K)]
    for qt, N, K in shapes:
        data = synth.weight_bytes(g, qt, N, K)
        qs = [torch.from_numpy(data).cuda() for _ in range(3)]
        dst = torch.empty((N, K), dtype=torch.float16, device="cuda")
        calls = [functools.partial(mq.mq_dequantize, qt, q, N, K, dst, None, stream) for q in qs] * 4
        t_us = _rotating_time_us(torch, calls, stream)
        byts = synth.nblocks(qt, N, K) * synth.BLOCK[qt][1] + 2 * N * K
        out[synth.TYPE_NAME[qt]] = {"N": N, "K": K, "us": t_us, "bytes": byts,
                                    "gbs": byts / (t_us * 1e-6) / 1e9,
                                    "frac_hbm": byts / (t_us * 1e-6) / 1e9 / P["hbm_gbs"]}
        del qs, dst
    mq.mq_stream_status()
    return out


if __name__ == "__main__":
    sys.exit(main())
