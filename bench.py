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

Printed: one JSON line with the contract keys plus
  roofline      the cached GEMM kernel against the measured dense peak: its
                time per step is its share of the kernel time in a traced
                pass (library trace events around every launch) times the
                untraced step time; the f16 matmul peak is re-measured in
                the same run;
  cpu_baseline  the CPU oracle (f64) on a bounded sample of the same layer,
                on all host cores and on one core, plus the oracle's
                decoders per format and its GEMM time per configuration;
  e2e           the same metric with host buffers: pinned-host inputs copied
                in and all outputs copied out inside the timed region;
  library_f16_layer  context: the same step through cuBLAS (torch.mm) on the
                same decoded f16 weights, f32 and f16 outputs;
  decode        the registration decoders (mq_register_weight of the 7
                weights back to back on a busy stream) against HBM bandwidth;
  decode_steady the decoders back to back on the 7B gate/down shapes and
                weights of the other formats at the gate's shape (HBM GB/s);
  small_m       fused vs cached over the small-M sweep, back to back over
                rotating weight copies (crossover, HBM GB/s);
  c2_llama3.1-8b_layer  the Llama-3.1-8B layer at M = 512: cached (K-padded
                caches and unpadded), fused and the M gate, per layer and
                per GEMM;
  c3_q8_0_pair  the Q8_0 pair: registration and steady decode, cached /
                fused / M gate over M = 1 .. 1024 with its crossover;
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

One GPU per run: with --gpus N > 1 (or under torchrun with more than one
rank) no rank touches a GPU and rank 0 prints a line that says so.
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
NOMINAL_F16_TFLOPS = 2250.0   # dense f16/bf16 tensor rate per GB300, vendor figure
NOMINAL_HBM_GBS = 7900.0      # HBM3e per GB300, vendor figure


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


def layer_decode_bytes(weights):
    """Algorithmic bytes of decoding the weights: blocks read + f16 written once."""
    return sum(synth.nblocks(w.qtype, w.N, w.K) * synth.BLOCK[w.qtype][1] + 2 * w.N * w.K for w in weights)


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

SINGLE_GPU_NOTE = ("single-GPU path: the library runs one GPU per process and nothing here launches it on "
                   "more than one GPU (the path shards by tokens or weight rows with no exchange; see replicas)")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle sample budget for cpu_baseline")
    ap.add_argument("--no-extras", action="store_true", help="skip e2e, the extra workloads and cpu_baseline")
    ap.add_argument("--clocks-out", default=None)
    ap.add_argument("--oracle-child", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_child:
        return oracle_child(args.oracle_child)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus > 1 or world > 1:
        # One GPU per run: no rank touches a GPU; rank 0 says so.
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": None, "unit": "TFLOP/s", "n_gpus": max(args.gpus, world),
                              "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
                              "config": {"workload": WORKLOAD, "M": M_TOKENS}, "skipped": SINGLE_GPU_NOTE}))
        return 0

    import torch
    import quantized_weight_prefill_gguf_gb300 as mq

    torch.cuda.set_device(0)
    P = peaks()
    weights, xs = synth.workload(WORKLOAD, seed=0)

    stream = torch.cuda.current_stream()
    qdev = [torch.from_numpy(w.data).cuda() for w in weights]
    torch.cuda.synchronize()

    # registration = one-time decode into the f16 caches, traced per weight
    # (the process's first decode launches: cold, see registration_decode)
    mq.mq_trace_enable(True)
    handles = [mq.mq_register_weight(w.qtype, q, w.N, w.K) for w, q in zip(weights, qdev)]
    torch.cuda.synchronize()
    dec = [r for r in mq.mq_trace_records() if r["kind"] == mq.MQ_TRACE_DECODE]
    mq.mq_trace_enable(False)
    decode_bytes = layer_decode_bytes(weights)
    decode_cold_ms = sum(r["ms_main"] for r in dec)

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
    clocks = ClockSampler(0, args.clocks_out)
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = mq.mq_launch_count()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        step(xdev)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = mq.mq_launch_count() - launches0
    clk = clocks.stop()
    mq.mq_stream_status()
    ms = ev0.elapsed_time(ev1) / args.steps

    # Kernel shares for the roofline: a separate pass with the library's
    # trace events around every launch (events between two launches end the
    # overlap that programmatic dependent launch gives, so the timed steps
    # above run without them; only the shares are taken from this pass).
    trace_steps = min(args.steps, 200)
    mq.mq_trace_enable(True)
    for _ in range(trace_steps):
        step(xdev)
    torch.cuda.synchronize()
    mq.mq_trace_enable(False)

    flops_step = layer_flops(weights, M_TOKENS)
    value = flops_step / (ms * 1e-3) / 1e12
    f16_peak = f16_matmul_peak(torch)

    # ---- roofline of the dominant kernel: the cached GEMM (k_gemm_cached*)
    recs = mq.mq_trace_records()
    gem = [r for r in recs if r["kind"] == mq.MQ_TRACE_GEMM_CACHED]
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
                             "gemm_us_traced": t_main * 1e3, "reduce_us_traced": t_aux * 1e3})
    # The GEMM kernel's time per step = its share of the traced kernel time
    # (GEMM + split-K reduce) x the untraced step time; all the step's FLOPs
    # are the GEMM kernel's (the reduce only adds partial planes).
    share = g_ms / (g_ms + red_ms) if g_ms > 0 else None
    kern_ms = share * ms if share else None
    if kern_ms is not None:
        assert kern_ms <= ms * (1 + 1e-9), "kernel time per step exceeds the step"
    achieved = flops_step / (kern_ms * 1e-3) / 1e12 if kern_ms else None
    traffic = None
    tp = os.path.join(ROOT, "profiles", "k_gemm_cached.qwen2.5-7b_layer.traffic.json")
    if os.path.exists(tp):
        with open(tp) as fh:
            rec = json.load(fh)
        # the counters only describe the kernel source they were taken from
        if rec.get("kernel_source_sha256") == cached_kernel_source_hash():
            traffic = rec.get("k_gemm_cached_bytes_per_launch")
    n_launch = max(1, len(gem) // max(1, trace_steps))
    roofline = {"bound": "tensor", "achieved": achieved, "peak": P["bf16_tflops"], "unit": "TFLOP/s",
                "frac": (achieved / P["bf16_tflops"]) if achieved else None, "traffic": traffic,
                "kernel": "k_gemm_cached_2sm / k_gemm_cached (tcgen05 f16 GEMM on the f16 cache)",
                "peak_kind": f"dense bf16 burst ({P['source']}); the f16 nominal rate equals bf16",
                "peak_f16_same_run": f16_peak,
                "frac_of_f16_same_run": (achieved / f16_peak) if achieved and f16_peak else None,
                "frac_of_sustained": (achieved / P["bf16_tflops_sustained"]) if achieved else None,
                "frac_of_nominal": (achieved / NOMINAL_F16_TFLOPS) if achieved else None,
                "nominal_note": f"{NOMINAL_F16_TFLOPS:.0f} TFLOP/s dense f16 per GB300 (vendor figure, not measured)",
                "step_frac": value / P["bf16_tflops"],
                "kernel_share_of_step": share, "kernel_ms_per_step": kern_ms,
                "launches_per_step": n_launch,
                "method": "achieved = the step's FLOPs / (GEMM kernel share of the traced kernel time x the "
                          "untraced ms_per_step); traffic = DRAM bytes per launch from one ncu capture",
                "traced_steps": trace_steps, "reduce_share_of_step": (1 - share) if share else None}

    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_TOKENS, "gemms": [w.name for w in weights],
                   "weights": "q/k/v/o/gate/up Q4_K, down Q6_K (seeded synthetic blocks, model shapes)",
                   "gflop_per_step": flops_step / 1e9,
                   "path": "mq_gemm_grouped (q|k|v, gate|up) + mq_gemm_auto -> cached (o, down)",
                   "l2": "inputs larger than L2: 466 MB of f16 weight caches per step vs 126 MB L2",
                   "parallelism": "one GPU"},
        "tok_per_s_per_layer": M_TOKENS / (ms * 1e-3),
        "tok_per_s_28_layer_gemms_only": M_TOKENS / (28 * ms * 1e-3),
        "frac_of_peak": value / P["bf16_tflops"],
        "roofline": roofline,
        "per_gemm": per_gemm,
        "gpu_launches": launches,
        "clocks": clk,
    }
    out["decode"] = registration_decode(mq, torch, stream, weights, qdev, P)
    out["decode"]["cold_ms"] = decode_cold_ms
    out["decode"]["cold_gbs"] = decode_bytes / (decode_cold_ms * 1e-3) / 1e9 if decode_cold_ms else None

    if not args.no_extras:
        out["e2e"] = e2e_run(mq, torch, weights, handles, xs, ys, stream, min(args.steps, 50), flops_step)
        out["library_f16_layer"] = library_layer(mq, torch, stream, weights, qdev, xdev, min(args.steps, 50),
                                                 flops_step, ms)
        out["small_m"] = small_m_sweep(mq, torch, stream, P)
        out["decode_steady"] = decode_steady(mq, torch, stream, P)
        out["c2_llama3.1-8b_layer"] = llama_layer(mq, torch, stream, P)
        out["c3_q8_0_pair"] = q8_pair(mq, torch, stream, P)
        out["more_formats"] = more_formats(mq, torch, stream, P)
        out["triangle"] = triangle(mq, torch, stream, weights, handles, qdev, xdev)
        out["row_pad"] = row_pad(mq, torch, stream)
        out["e4m3"] = e4m3_layer(mq, torch, stream, weights, qdev, xdev, ys, P, min(args.steps, 400), flops_step)
        out["cpu_baseline"] = cpu_baseline(weights, xs, args.cpu_seconds)
    for h in handles:
        h.release()
    print(json.dumps(out))
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


def e2e_run(mq, torch, weights, handles, xs, ys, stream, steps, flops_step):
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
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for t in range(steps):
        step(t)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": flops_step / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "copies": "pinned host <-> device on two copy streams, double-buffered device X and Y"}


def _rotating_time_us(torch, fns, stream, reps=5):
    """Median per-call device time of the calls in `fns`, issued back to back
    on `stream` (CUDA events around the whole run of calls).  A sleep kernel
    ahead of the first event keeps the stream busy while the host enqueues
    the calls: an event recorded on an idle GPU would start the clock before
    the host has submitted the first call, adding its launch latency to the
    run."""
    for fn in fns:
        fn()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for fn in fns:
        fn()
    host_s = time.perf_counter() - t0
    torch.cuda.synchronize()
    busy_cycles = int(max(50e-6, 2.0 * host_s) * 2.5e9)
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(busy_cycles)
        a.record(stream)
        for fn in fns:
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3 / len(fns))
    return statistics.median(ts)


def _paths_rotating(mq, torch, stream, P, w, x_all, ms, paths=("fused", "cached")):
    """Rows {name, M, copies, <path>_us/_tflops/_gbs/_frac_hbm} for weight w
    at each M and each path of `paths` ("fused": mq_gemm_fused, "cached":
    mq_gemm, "cached_nokpad": mq_gemm on copies registered with
    MQ_REG_NO_KPAD, "auto": mq_gemm_auto): per-call time of calls issued back
    to back over R registered copies of the weight, R chosen so the weights
    touched (raw blocks for fused, f16 caches for cached) exceed 400 MB, three
    times the L2: every call streams its weight from HBM, as in a layer stack,
    and the launch gap between calls is included.  "auto" is charged the
    bytes of the path the M gate picks."""
    raw_bytes = synth.nblocks(w.qtype, w.N, w.K) * synth.BLOCK[w.qtype][1]
    R = max(3, -(-(400 << 20) // raw_bytes))
    qs = [torch.from_numpy(w.data).cuda() for _ in range(R)]
    hs = [mq.mq_register_weight(w.qtype, q, w.N, w.K) for q in qs]
    hs_nokpad = ([mq.mq_register_weight(w.qtype, q, w.N, w.K, flags=mq.MQ_REG_NO_KPAD) for q in qs]
                 if "cached_nokpad" in paths else [])
    fns = {"fused": (mq.mq_gemm_fused, hs), "cached": (mq.mq_gemm, hs), "cached_nokpad": (mq.mq_gemm, hs_nokpad),
           "auto": (mq.mq_gemm_auto, hs)}
    gate = mq.mq_get_m_gate()
    rows = []
    for M in ms:
        x = x_all[:M].contiguous()
        y = torch.empty((M, w.N), dtype=torch.float32, device="cuda")
        row = {"name": w.name, "M": M, "copies": R}
        for path in paths:
            fn, hh = fns[path]
            calls = [functools.partial(fn, x, h, y, M, stream) for h in hh]
            t_us = _rotating_time_us(torch, calls, stream)
            fused_bytes = path == "fused" or (path == "auto" and M < gate)
            wbytes = raw_bytes if fused_bytes else 2 * w.N * w.K
            byts = wbytes + 2 * M * w.K + 4 * M * w.N
            row[path + "_us"] = t_us
            row[path + "_tflops"] = 2.0 * M * w.N * w.K / (t_us * 1e-6) / 1e12
            row[path + "_gbs"] = byts / (t_us * 1e-6) / 1e9
            row[path + "_frac_hbm"] = row[path + "_gbs"] / P["hbm_gbs"]
        if "auto" in paths:
            row["auto_took"] = "fused" if M < gate else "cached"
        rows.append(row)
    mq.mq_stream_status()
    for h in hs + hs_nokpad:
        h.release()
    del qs
    return rows


def _fused_vs_cached(mq, torch, stream, P, w, x_all, ms):
    return _paths_rotating(mq, torch, stream, P, w, x_all, ms, ("fused", "cached"))


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
    # Hot-L2 reference: the same single registered copy called back to back,
    # so its raw blocks (38 / 56 MB) stay in the 126 MB L2 between calls.
    hot = []
    for w in weights:
        if w.name == "up":
            continue
        q = torch.from_numpy(w.data).cuda()
        h = mq.mq_register_weight(w.qtype, q, w.N, w.K, flags=mq.MQ_REG_NO_CACHE)
        x_all = torch.from_numpy(xs[w.K]).cuda()
        for M in (1, 32):
            x = x_all[:M].contiguous()
            y = torch.empty((M, w.N), dtype=torch.float32, device="cuda")
            t_us = _rotating_time_us(torch, [functools.partial(mq.mq_gemm_fused, x, h, y, M, stream)] * 8, stream)
            hot.append({"name": w.name, "M": M, "fused_us_hot_l2": t_us})
        mq.mq_stream_status()
        h.release()
    return {"rows": res, "cached_wins_from_M": cross, "gate_in_use": mq.mq_get_m_gate(), "hot_l2": hot,
            "method": "back to back over rotating weight copies (> 3x L2), per-call average including launch gaps; "
                      "hot_l2: one copy called back to back (labelled: its weight stays in L2)"}


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
    rel = float(torch.linalg.norm(ys[gi] - ys_f16[gi]) / torch.linalg.norm(ys_f16[gi]))
    mq.mq_stream_status()
    for h in hs:
        h.release()
    small = _e4m3_small_m(mq, torch, stream, weights[gi], qdev[gi], xdev, P)
    return {"ms_per_step": ms, "tflops": flops_step / (ms * 1e-3) / 1e12, "steps": steps, "small_m": small,
            "kernel": {"name": "k_gemm_e4m3", "achieved_tflops": achieved, "peak_tflops": peak8,
                       "peak_note": "8-bit dense = 2 x the measured bf16 burst peak (the nominal fp8:bf16 ratio)",
                       "frac": achieved / peak8 if achieved else None},
            "rel_distance_to_f16_gate": rel,
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


def library_layer(mq, torch, stream, weights, qdev, xdev, steps, flops_step, ms_ours):
    """Context, not a product path: the same layer step through a library
    GEMM (torch.mm, i.e. cuBLAS) on the same f16 operands -- the weights
    decoded by mq_dequantize into plain N x K f16 tensors, concatenated per
    launch group exactly as the library's grouped launches see them -- timed
    like the step (events around `steps` back-to-back steps after warm-up;
    the 466 MB of f16 weights per step exceed L2).  Two output types: f32
    (the library's own output type; torch.mm with out_dtype, where this
    torch has it) and f16."""
    w16 = []
    for w, q in zip(weights, qdev):
        t = torch.empty((w.N, w.K), dtype=torch.float16, device="cuda")
        mq.mq_dequantize(w.qtype, q, w.N, w.K, t, stream=stream)
        w16.append(t)
    by_name = {w.name: i for i, w in enumerate(weights)}
    groups = []
    for grp in LAUNCH_GROUPS:
        idx = [by_name[n] for n in grp]
        wt = torch.cat([w16[i] for i in idx], 0) if len(idx) > 1 else w16[idx[0]]
        groups.append((xdev[weights[idx[0]].K], wt))
    del w16
    out = {"ms_per_step_ours": ms_ours,
           "note": "cuBLAS through torch.mm on the decoded f16 weights, one GEMM per launch group "
                   "(q|k|v, o, gate|up, down); a comparison only, never the library's path"}
    for label, dt in (("f32_out", torch.float32), ("f16_out", torch.float16)):
        ys = [torch.empty((x.shape[0], wt.shape[0]), dtype=dt, device="cuda") for x, wt in groups]

        def step():
            for (x, wt), y in zip(groups, ys):
                if dt == torch.float32:
                    torch.mm(x, wt.t(), out_dtype=torch.float32, out=y)
                else:
                    torch.mm(x, wt.t(), out=y)
        try:
            for _ in range(3):
                step()
            torch.cuda.synchronize()
        except (RuntimeError, TypeError) as e:
            out[label] = {"unavailable": str(e).splitlines()[0][:160]}
            continue
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / steps
        out[label] = {"ms_per_step": t, "tflops": flops_step / (t * 1e-3) / 1e12,
                      "ours_over_library": t / ms_ours}
        del ys
    del groups
    torch.cuda.empty_cache()
    return out


def f16_matmul_peak(torch, n=8192, reps=10):
    """Dense f16 tensor-core rate measured in this run: torch.matmul (a
    library GEMM, used only as the roofline's denominator) on n x n x n f16
    operands, best of `reps` single calls after warm-up (burst clocks)."""
    a = torch.randn(n, n, device="cuda", dtype=torch.float16)
    b = torch.randn(n, n, device="cuda", dtype=torch.float16)
    for _ in range(3):
        torch.matmul(a, b)
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        best = t if best is None else min(best, t)
    del a, b
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


def registration_decode(mq, torch, stream, weights, qdev, P):
    """mq_register_weight of the given weights as one sequence, the product's
    decode entry point: each call allocates the f16 cache and enqueues the
    decoder.  Timed on the device with CUDA events around the whole
    sequence while a sleep kernel keeps the stream busy until the host has
    issued every call, so neither host launch latency nor an idle GPU enters
    the window (a single event-timed call on an idle GPU includes the host's
    launch latency).  A first, untimed pass loads the decode kernels.  Best
    of three, with no events between the calls (an event between two
    launches ends their programmatic overlap); `kernel_ms` sums the decode
    kernels' own durations from the library's trace events in a separate
    pass."""
    nbytes = layer_decode_bytes(weights)

    def register_all():
        return [mq.mq_register_weight(w.qtype, q, w.N, w.K, stream=stream) for w, q in zip(weights, qdev)]

    t0 = time.perf_counter()
    hs = register_all()
    torch.cuda.synchronize()
    host_s = time.perf_counter() - t0
    for h in hs:
        h.release()
    busy_s = max(0.002, 4.0 * host_s)
    best = None
    for _ in range(3):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(busy_s * 2.5e9))
        e0.record(stream)
        t0 = time.perf_counter()
        hs = register_all()
        issue_s = time.perf_counter() - t0
        e1.record(stream)
        torch.cuda.synchronize()
        seq_ms = e0.elapsed_time(e1)
        for h in hs:
            h.release()
        if best is None or seq_ms < best["ms"]:
            best = {"ms": seq_ms, "issue_ms": issue_s * 1e3, "busy_ms": busy_s * 1e3}
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(busy_s * 2.5e9))
    mq.mq_trace_enable(True)
    hs = register_all()
    torch.cuda.synchronize()
    kern_ms = sum(r["ms_main"] for r in mq.mq_trace_records() if r["kind"] == mq.MQ_TRACE_DECODE)
    mq.mq_trace_enable(False)
    for h in hs:
        h.release()
    gbs = nbytes / (best["ms"] * 1e-3) / 1e9
    best.update({"bytes": nbytes, "gbs": gbs, "frac_hbm": gbs / P["hbm_gbs"],
                 "frac_hbm_nominal": gbs / NOMINAL_HBM_GBS, "kernel_ms_traced": kern_ms,
                 "kernel_gbs_traced": nbytes / (kern_ms * 1e-3) / 1e9 if kern_ms else None,
                 "stream_stayed_busy": best["issue_ms"] < best["busy_ms"],
                 "weights": len(weights),
                 "note": "mq_register_weight of every weight back to back (blocks read + f16 written once), "
                         "device-timed on a busy stream; kernel_*_traced: events around each decode (no "
                         "launch overlap); cold_* = the process's first registration, event-timed per call on "
                         "an idle GPU (kernel loading and host launch latency included)"})
    return best


LLAMA_M = 512


def llama_layer(mq, torch, stream, P):
    """Config c2: the Llama-3.1-8B-shaped layer (all Q4_K; K = 4096 and
    14336, so the f16 caches are K-padded by one 128-byte line) at M = 512.
    Per layer (the layer's four launch groups back to back, rotating over
    R copies of the layer: > 400 MB of raw blocks touched): cached (padded
    caches), cached without the pad (MQ_REG_NO_KPAD), fused (raw blocks)
    and the M gate (auto).  Per GEMM shape: the same paths on single
    weights (_paths_rotating)."""
    clocks = ClockSampler(0)
    clocks.start()
    weights, xs = synth.workload("llama3.1-8b_layer", seed=0)
    M = LLAMA_M
    xdev = {K: torch.from_numpy(x[:M]).cuda() for K, x in xs.items()}
    raw = sum(w.data.size for w in weights)
    R = max(2, -(-(400 << 20) // raw))
    copies = []
    for _ in range(R):
        q = [torch.from_numpy(w.data).cuda() for w in weights]
        copies.append({"q": q,
                       "cached": [mq.mq_register_weight(w.qtype, qq, w.N, w.K) for w, qq in zip(weights, q)],
                       "cached_nokpad": [mq.mq_register_weight(w.qtype, qq, w.N, w.K, flags=mq.MQ_REG_NO_KPAD)
                                         for w, qq in zip(weights, q)],
                       "fused": [mq.mq_register_weight(w.qtype, qq, w.N, w.K, flags=mq.MQ_REG_NO_CACHE)
                                 for w, qq in zip(weights, q)]})
    ys = [torch.empty((M, w.N), dtype=torch.float32, device="cuda") for w in weights]
    by = {w.name: i for i, w in enumerate(weights)}
    groups = [[by[n] for n in grp] for grp in LAUNCH_GROUPS]
    single = {"cached": mq.mq_gemm, "cached_nokpad": mq.mq_gemm, "fused": mq.mq_gemm_fused, "auto": mq.mq_gemm_auto}
    grouped = {"cached": mq.mq_gemm_grouped, "cached_nokpad": mq.mq_gemm_grouped,
               "fused": mq.mq_gemm_fused_grouped, "auto": mq.mq_gemm_auto_grouped}

    def layer_fn(c, mode):
        hs = c["cached" if mode == "auto" else mode]

        def run():
            for idx in groups:
                x = xdev[weights[idx[0]].K]
                if len(idx) == 1:
                    single[mode](x, hs[idx[0]], ys[idx[0]], M, stream)
                else:
                    grouped[mode](x, [hs[i] for i in idx], [ys[i] for i in idx], M, stream)
        return run

    flops = layer_flops(weights, M)
    layer = {}
    for mode in ("cached", "cached_nokpad", "fused", "auto"):
        t_us = _rotating_time_us(torch, [layer_fn(c, mode) for c in copies], stream)
        layer[mode + "_us"] = t_us
        layer[mode + "_tflops"] = flops / (t_us * 1e-6) / 1e12
    mq.mq_stream_status()
    ldk = copies[0]["cached"][0].info()[2]
    for c in copies:
        for h in c["cached"] + c["cached_nokpad"] + c["fused"]:
            h.release()
    del copies
    per_gemm = []
    for name in ("q", "k", "gate", "down"):
        w = weights[by[name]]
        per_gemm += _paths_rotating(mq, torch, stream, P, w, xdev[w.K], [M],
                                    ("cached", "cached_nokpad", "fused", "auto"))
    clk = clocks.stop()
    return {"M": M, "gflop_per_layer": flops / 1e9, "ldk_padded": ldk, "layer": layer, "layer_copies": R,
            "per_gemm": per_gemm, "gate_in_use": mq.mq_get_m_gate(), "clocks": clk,
            "method": "layer = four launches (q|k|v and gate|up grouped, o, down) back to back over R layer "
                      "copies; per GEMM as small_m (rotating copies, > 400 MB touched)"}


def q8_pair(mq, torch, stream, P):
    """Config c3: Q8_0 weights 3584 x 18944 and 18944 x 3584 (34-byte blocks,
    2-byte aligned; K = 18944 and 3584 are not multiples of 1024, so the
    caches are not padded).  Decode through mq_register_weight (busy-stream
    sequence) and mq_dequantize back to back; GEMMs through the cached path,
    the fused path and the M gate at M in {1, 8, 32, 128, 129, 192, 256, 512, 1024}
    (M = 128 and 1024 are the configuration's own), rotating copies."""
    clocks = ClockSampler(0)
    clocks.start()
    weights, xs = synth.workload("q8_0_pair", seed=0)
    qdev = [torch.from_numpy(w.data).cuda() for w in weights]
    reg = registration_decode(mq, torch, stream, weights, qdev, P)
    steady = {}
    for w, q in zip(weights, qdev):
        qs = [q] + [q.clone() for _ in range(2)]
        dst = torch.empty((w.N, w.K), dtype=torch.float16, device="cuda")
        calls = [functools.partial(mq.mq_dequantize, w.qtype, qq, w.N, w.K, dst, None, stream) for qq in qs] * 4
        t_us = _rotating_time_us(torch, calls, stream)
        byts = layer_decode_bytes([w])
        steady[w.name] = {"N": w.N, "K": w.K, "us": t_us, "gbs": byts / (t_us * 1e-6) / 1e9,
                          "frac_hbm": byts / (t_us * 1e-6) / 1e9 / P["hbm_gbs"]}
        del qs, dst
    rows = []
    for w in weights:
        x_all = torch.from_numpy(xs[w.K]).cuda()
        rows += _paths_rotating(mq, torch, stream, P, w, x_all, [1, 8, 32, 128, 129, 192, 256, 512, 1024],
                                ("fused", "cached", "auto"))
    cross = {}
    for w in weights:
        ms_ = [r["M"] for r in rows if r["name"] == w.name and r["cached_us"] <= r["fused_us"]]
        cross[w.name] = min(ms_) if ms_ else None
    flops_pair = {M: sum(2.0 * M * w.N * w.K for w in weights) for M in (128, 1024)}
    headline = {}
    for M in (128, 1024):
        sel = [r for r in rows if r["M"] == M]
        headline[f"M{M}"] = {p + "_tflops_pair": flops_pair[M] / (sum(r[p + "_us"] for r in sel) * 1e-6) / 1e12
                             for p in ("fused", "cached", "auto")}
    clk = clocks.stop()
    return {"decode_registration": reg, "decode_steady": steady, "rows": rows, "headline": headline,
            "cached_wins_from_M": cross, "gate_in_use": mq.mq_get_m_gate(), "clocks": clk}


def oracle_child(tokens: int) -> int:
    """Child process of cpu_baseline: time the oracle's f64 GEMM over the 7B
    layer for `tokens` tokens with the OpenMP thread count this process was
    started with (OMP_NUM_THREADS); print one JSON line."""
    import oracle
    orc = oracle.load()
    weights, xs = synth.workload(WORKLOAD, seed=0)
    W16 = [orc.decode_matrix(w.qtype, w.data, w.N, w.K) for w in weights]
    t0 = time.perf_counter()
    for w, W in zip(weights, W16):
        orc.gemm_f64(xs[w.K][:tokens].view(np.uint16), W)
    secs = time.perf_counter() - t0
    print(json.dumps({"tokens": tokens, "secs": secs, "threads": orc.num_threads(),
                      "tflops": layer_flops(weights, tokens) / secs / 1e12}))
    return 0


def cpu_baseline(weights, xs, budget_s):
    """The oracle as it stands, timed on this host's cores: the 7B layer's f64
    GEMM on a token sample sized to about budget_s seconds with every core
    (the headline value), the same on one core (a child process with
    OMP_NUM_THREADS=1, a smaller sample), the oracle's decoders per format
    (best of 3, GB/s of blocks read + f16 written) and its GEMM time per
    configuration, extrapolated linearly in M from a token sample."""
    import oracle
    orc = oracle.load()
    tf, tokens, secs, dsec, threads = oracle_cpu_run(weights, xs, budget_s)
    res = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{tokens} of {M_TOKENS} tokens through all 7 GEMMs of the 7B layer (f64, {secs:.1f} s) "
                     f"on all {threads} threads; the oracle's decode of the 7 weights took {dsec:.1f} s before",
           "cores_all": threads}
    per_tok_1 = secs / tokens * threads   # rough single-core cost per token, sizes the child's sample
    t1 = int(max(1, min(M_TOKENS, 8.0 / max(per_tok_1, 1e-9))))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", str(t1)], env=env,
                           capture_output=True, text=True, timeout=300)
        child = json.loads(r.stdout.strip().splitlines()[-1])
        res["value_1core"] = child["tflops"]
        res["sample_1core"] = f"{child['tokens']} tokens, {child['secs']:.1f} s, {child['threads']} thread"
    except (subprocess.SubprocessError, ValueError, IndexError, KeyError) as e:
        res["value_1core"] = None
        res["sample_1core"] = f"failed: {e}"
    g = synth.rng(5)
    dec = {}
    for qt, N, K in ((synth.Q4_K, 18944, 3584), (synth.Q6_K, 3584, 18944), (synth.Q8_0, 18944, 3584)):
        data = synth.weight_bytes(g, qt, N, K)
        best = None
        for _ in range(3):
            t0 = time.perf_counter()
            orc.decode_matrix(qt, data, N, K)
            t = time.perf_counter() - t0
            best = t if best is None else min(best, t)
        dec[synth.TYPE_NAME[qt]] = {"N": N, "K": K, "s": best,
                                    "gbs": layer_decode_bytes([synth.Weight("w", qt, N, K, data)]) / best / 1e9}
    res["decode_gbs"] = dec
    per_cfg = {"qwen2.5-7b_layer": {"M2048_s_est": secs / tokens * M_TOKENS, "sample_tokens": tokens}}
    for name in ("q4k_896", "llama3.1-8b_layer", "q8_0_pair"):
        ws, xx = synth.workload(name, seed=0)
        W16 = [orc.decode_matrix(w.qtype, w.data, w.N, w.K) for w in ws]
        for M in synth.WORKLOADS[name][1]:
            t0 = time.perf_counter()
            for w, W in zip(ws, W16):
                orc.gemm_f64(xx[w.K][:M].view(np.uint16), W)
            per_cfg.setdefault(name, {})[f"M{M}_s"] = time.perf_counter() - t0
    res["gemm_s_per_config"] = per_cfg
    res["gemm_s_note"] = ("f64 GEMM of every weight of the configuration at its full M, all threads, one run; "
                          "the 7B layer's from the token sample above, scaled to M = 2048 (linear in M)")
    return res


if __name__ == "__main__":
    sys.exit(main())
