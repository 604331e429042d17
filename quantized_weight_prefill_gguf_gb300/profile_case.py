"""Run one GEMM or decode case a few times, for a profiler (ncu) to capture.

    python -m quantized_weight_prefill_gguf_gb300.profile_case \
        --case fused --type q4_K --N 18944 --K 3584 --M 32 --reps 3

Cases: cached (mq_gemm), fused (mq_gemm_fused), decode (mq_dequantize),
e4m3 (mq_gemm_e4m3 on activations quantized once before), quant
(mq_quantize_e4m3 of the M x K activations).  --group G (cached, fused): G
weights of the shape in one mq_gemm_grouped / mq_gemm_fused_grouped call.
--library (cached, one weight): after the library's calls, the same GEMM
through cuBLAS (torch.mm with an f32 output) on the weight decoded to f16 by
mq_dequantize, --reps times, for a side-by-side capture of the two kernels;
a comparison only.  Inputs are the seeded synthetic blocks of the given
shape.  Prints the
device time of each call from the library's trace events (not valid under a
profiler, which serialises and replays kernels).
"""
from __future__ import annotations

import argparse

import torch

import quantized_weight_prefill_gguf_gb300 as mq
from quantized_weight_prefill_gguf_gb300 import synth

TYPES = {synth.TYPE_NAME[t]: t for t in synth.BLOCK}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=["cached", "fused", "decode", "e4m3", "quant"], required=True)
    ap.add_argument("--type", choices=sorted(TYPES), default="q4_K")
    ap.add_argument("--N", type=int, required=True)
    ap.add_argument("--K", type=int, required=True)
    ap.add_argument("--M", type=int, default=32)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--group", type=int, default=1)
    ap.add_argument("--library", action="store_true")
    args = ap.parse_args(argv)
    if args.library and (args.case != "cached" or args.group != 1):
        ap.error("--library applies to --case cached with one weight")

    qtype = TYPES[args.type]
    g = synth.rng(args.seed)
    data = synth.weight_bytes(g, qtype, args.N, args.K)
    q = torch.from_numpy(data).cuda()
    if args.case == "decode":
        out = torch.empty((args.N, args.K), dtype=torch.float16, device="cuda")
        fn = lambda: mq.mq_dequantize(qtype, q, args.N, args.K, out)  # noqa: E731
    elif args.case in ("e4m3", "quant"):
        h = mq.mq_register_weight(qtype, q, args.N, args.K, flags=mq.MQ_REG_E4M3)
        x = torch.from_numpy(synth.activations(g, args.M, args.K)).cuda()
        x8 = torch.empty((args.M, args.K), dtype=torch.uint8, device="cuda")
        sx = torch.empty(args.M, dtype=torch.float32, device="cuda")
        mq.mq_quantize_e4m3(x, x8, sx)
        y = torch.empty((args.M, args.N), dtype=torch.float32, device="cuda")
        if args.case == "quant":
            fn = lambda: mq.mq_quantize_e4m3(x, x8, sx)  # noqa: E731
        else:
            fn = lambda: mq.mq_gemm_e4m3(x8, sx, h, y, args.M)  # noqa: E731
    elif args.group > 1:
        flags = mq.MQ_REG_NO_CACHE if args.case == "fused" else 0
        qs = [q] + [torch.from_numpy(synth.weight_bytes(g, qtype, args.N, args.K)).cuda()
                    for _ in range(args.group - 1)]
        hs = [mq.mq_register_weight(qtype, qi, args.N, args.K, flags=flags) for qi in qs]
        x = torch.from_numpy(synth.activations(g, args.M, args.K)).cuda()
        ys = [torch.empty((args.M, args.N), dtype=torch.float32, device="cuda") for _ in hs]
        call = mq.mq_gemm_fused_grouped if args.case == "fused" else mq.mq_gemm_grouped
        fn = lambda: call(x, hs, ys, args.M)  # noqa: E731
    else:
        flags = mq.MQ_REG_NO_CACHE if args.case == "fused" else 0
        h = mq.mq_register_weight(qtype, q, args.N, args.K, flags=flags)
        x = torch.from_numpy(synth.activations(g, args.M, args.K)).cuda()
        y = torch.empty((args.M, args.N), dtype=torch.float32, device="cuda")
        call = mq.mq_gemm_fused if args.case == "fused" else mq.mq_gemm
        fn = lambda: call(x, h, y, args.M)  # noqa: E731
    torch.cuda.synchronize()
    mq.mq_trace_enable(True)
    for _ in range(args.reps):
        fn()
    torch.cuda.synchronize()
    mq.mq_stream_status()
    for r in mq.mq_trace_records():
        print(f"{args.case} {args.type} M={args.M} N={args.N}x{args.group} K={args.K}: "
              f"{r['ms_main'] * 1e3:.1f} us (+ reduce {r['ms_aux'] * 1e3:.1f} us)")
    if args.library:
        w16 = torch.empty((args.N, args.K), dtype=torch.float16, device="cuda")
        mq.mq_dequantize(qtype, q, args.N, args.K, w16)
        y_lib = torch.empty_like(y)
        for _ in range(args.reps):
            torch.mm(x, w16.t(), out_dtype=torch.float32, out=y_lib)
        torch.cuda.synchronize()
        print(f"library (torch.mm, f32 out) on the same f16 weight: max |difference| "
              f"{float((y - y_lib).abs().max()):.3g}")
    mq.mq_trace_enable(False)


if __name__ == "__main__":
    main()
