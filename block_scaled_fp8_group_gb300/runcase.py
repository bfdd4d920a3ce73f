"""Runs one GEMM (or linear) problem a few times -- the small, self-contained
command the profiler captures.

    python -m block_scaled_fp8_group_gb300.runcase --m 8 --n 18432 --k 7168 \
        --fmt ue8m0 --iters 3 [--variant swap/16/0[/grid/mma_scale]] [--op gemm|linear|quant]
    python -m block_scaled_fp8_group_gb300.runcase --m 8 --n 18432 --k 7168 \
        --op rowwise --code int8 --iters 3 [--variant swap/16/1]
    python -m block_scaled_fp8_group_gb300.runcase --m 2048 --n 7168 --k 18432 \
        --op int8block --iters 2
    python -m block_scaled_fp8_group_gb300.runcase --m 0 --n 4096 --k 7168 \
        --op grouped --tokens 128 --iters 2

Inputs are the decode-sweep distributions from ``synth`` (bf16 N(0,1) with 1%
outlier channels, bf16 N(0,0.02) weights), quantised on the GPU.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import fp8bq, synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--m", type=int, required=True)
    ap.add_argument("--n", type=int, required=True)
    ap.add_argument("--k", type=int, required=True)
    ap.add_argument("--fmt", default="ue8m0", choices=("fp32", "ue8m0"))
    ap.add_argument("--out", default="bf16", choices=("bf16", "fp16", "fp32"))
    ap.add_argument("--op", default="gemm",
                    choices=("gemm", "linear", "quant", "rowwise", "int8block", "grouped"))
    ap.add_argument("--tokens", type=int, default=128,
                    help="--op grouped: tokens routed top-8 over 32 local experts of 256 "
                         "(--n/--k: one expert's projection)")
    ap.add_argument("--code", default="e4m3", choices=("e4m3", "int8"),
                    help="--op rowwise: per-token x per-channel codes")
    ap.add_argument("--variant", default=None,
                    help="kind/block_n/split[/grid[/mma_scale]] (default: the table's)")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--time", action="store_true",
                    help="--op quant: also print the mean time of 50 back-to-back launches "
                         "over input copies larger than the L2 (CUDA events)")
    args = ap.parse_args()
    dev = torch.device("cuda")
    out_dt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[args.out]
    x = torch.from_numpy(synth.act_decode(args.m, args.k).view(np.int16)).view(
        torch.bfloat16).to(dev)
    if args.op == "quant":
        for _ in range(args.iters):
            fp8bq.fp8bq_quant_act(x, args.fmt)
        torch.cuda.synchronize()
        if args.time:
            time_quant(x, args.fmt)
        return
    if args.op == "grouped":
        # the MoE workload's grouped GEMM: E experts, counts from seeded routing
        E = synth.MOE_E_LOCAL
        counts = synth.moe_counts(E, args.tokens)
        M_max = int((counts.max() + 3) // 4 * 4)
        xg = torch.from_numpy(synth.moe_act(E, M_max, args.k).view(np.int16)).view(
            torch.bfloat16).to(dev)
        wb = synth.moe_weight_bf16(E, args.n, args.k)
        wq = torch.empty((E, args.n, args.k), dtype=torch.uint8, device=dev)
        ws = torch.empty((E, args.n // 128, args.k // 128), dtype=torch.float32, device=dev)
        for e in range(E):
            wd = torch.from_numpy(wb[e].view(np.int16)).view(torch.bfloat16).to(dev)
            fp8bq.fp8bq_quant_weight(wd, args.fmt, q=wq[e], s=ws[e])
        aq, as_ = fp8bq.fp8bq_quant_act(xg, args.fmt)
        cnt = torch.from_numpy(counts).to(dev)
        for _ in range(args.iters):
            fp8bq.fp8bq_grouped_gemm(aq, as_, wq, ws, cnt, fmt=args.fmt, out_dtype=out_dt)
        torch.cuda.synchronize()
        if fp8bq.fp8bq_device_status() != 0:
            raise SystemExit("device wait timed out")
        return
    w = torch.from_numpy(synth.weight_bf16(args.n, args.k).view(np.int16)).view(
        torch.bfloat16).to(dev)
    v = None
    if args.variant:
        parts = args.variant.split("/")
        v = fp8bq.make_variant(parts[0], int(parts[1]), int(parts[2]),
                               int(parts[3]) if len(parts) > 3 else 0,
                               int(parts[4]) if len(parts) > 4 else 0)
    if args.op == "int8block":
        # block INT8: 1x128 activation groups, 128x128 weight blocks
        xa = torch.from_numpy(synth.act_prefill(args.m, args.k).view(np.int16)).view(
            torch.bfloat16).to(dev)
        aq, as_ = fp8bq.fp8bq_quant_act_int8(xa)
        wq, ws = fp8bq.fp8bq_quant_weight_int8(w)
        for _ in range(args.iters):
            fp8bq.fp8bq_gemm_int8_block(aq, as_, wq, ws, out_dt, variant=v)
        torch.cuda.synchronize()
        if fp8bq.fp8bq_device_status() != 0:
            raise SystemExit("device wait timed out")
        return
    if args.op == "rowwise":
        wq, ws = fp8bq.fp8bq_quant_rows(w, args.code)
        aq, as_ = fp8bq.fp8bq_quant_rows(x, args.code)
        for _ in range(args.iters):
            fp8bq.fp8bq_gemm_rowwise(aq, as_, wq, ws, args.code, out_dt, variant=v)
        torch.cuda.synchronize()
        if fp8bq.fp8bq_device_status() != 0:
            raise SystemExit("device wait timed out")
        return
    wq, ws = fp8bq.fp8bq_quant_weight(w, args.fmt)
    aq, as_ = fp8bq.fp8bq_quant_act(x, args.fmt)
    for _ in range(args.iters):
        if args.op == "linear":
            fp8bq.fp8bq_linear(x, wq, ws, fmt=args.fmt, out_dtype=out_dt)
        elif v is not None:
            fp8bq.fp8bq_gemm_variant(aq, as_, wq, ws, v, fmt=args.fmt, out_dtype=out_dt)
        else:
            fp8bq.fp8bq_gemm(aq, as_, wq, ws, fmt=args.fmt, out_dtype=out_dt)
    torch.cuda.synchronize()
    if fp8bq.fp8bq_device_status() != 0:
        raise SystemExit("device wait timed out")


def time_quant(x, fmt, launches=50):
    """Mean device time of the activation quant: `launches` back-to-back
    launches captured in a CUDA graph (no host time between them) over
    rotated input copies that together exceed the 129 MB L2 (inputs smaller
    than 2 MB rotate through 64 copies and stay in L2: launch-bound sizes).
    Algorithmic bandwidth: 2 B in + 1 B out per element, plus the scales."""
    M, K = x.shape
    n = min(64, max(2, 1 + -(-(256 << 20) // (2 * M * K))))
    copies = [x] + [x.clone() for _ in range(n - 1)]
    qs = [fp8bq.fp8bq_quant_act(c, fmt) for c in copies]
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(launches):
                j = i % len(copies)
                fp8bq.fp8bq_quant_act(copies[j], fmt, q=qs[j][0], s=qs[j][1])
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    best = None
    for _ in range(3):
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        us = a.elapsed_time(b) * 1e3 / launches
        best = us if best is None else min(best, us)
    scale_bytes = qs[0][1].numel() * qs[0][1].element_size()
    byt = 3 * M * K + scale_bytes
    print(f"quant {fmt} M={M} K={K}: {best:.2f} us, {byt / best / 1e3:.1f} GB/s algorithmic "
          f"({len(copies)} input copies, {launches} launches in a graph, best of 3)")


if __name__ == "__main__":
    main()
