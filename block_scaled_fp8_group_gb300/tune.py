"""Builds the per-shape variant table by measurement ("vLLM 量化 Kernel 配置机制"
§3: per (N, K, device, dtype) and per point of the M grid, time every candidate
kernel configuration and keep the fastest).

    python -m block_scaled_fp8_group_gb300.tune \
        --sets small,decode,prefill,full,rowwise,rowwise_int8,block_int8,moe \
        [--out block_scaled_fp8_group_gb300/tables/<device>.tbl]

Candidates per M: swap-AB with token tiles 16..128 (and 64 weight rows per
tile for token tiles up to 32) and the normal
orientation with 128/256-wide weight tiles, each with stream-K (split 0),
no split, and a few fixed K splits; with UE8M0 scales and K % 512 == 0 every
candidate with 128-row tiles also runs with the scales applied by the
block-scaled MMA (mma_scale 1).  The INT8 sets ("ri8", "bi8") time both
INT8 kernels: the warp-level int8 MMA (mma_scale 0, token tiles from 8) and
the two e4m3 planes on the FP8 MMA (mma_scale 1).  The grouped set ("moe")
times the grouped GEMM over the MoE workload's 32 local experts and keys its
entries ("gue8m0") by the rows per expert.  Each candidate is timed on cold weights
(a rotation of weight copies larger than L2) as the mean of a batch of
back-to-back launches queued behind a GPU sleep, so launch gaps do not count
host time.  Lines of the table file: N K fmt out M kind block_n split grid
mma_scale.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import time

import numpy as np
import torch

from . import fp8bq, synth

HERE = os.path.dirname(os.path.abspath(__file__))
L2_BYTES = 160 << 20  # rotate through more than the L2 holds

SETS = {
    # (N, K, fmt, out dtype, M grid)
    "small": [(1536, 1536, "fp32", "bf16", (16,))],
    "decode": [(n, k, "ue8m0", "bf16", synth.DECODE_M) for n, k in synth.DECODE_NK],
    "prefill": [(n, k, "fp32", o, synth.PREFILL_M) for n, k in synth.PREFILL_NK
                for o in ("bf16", "fp32")],
    "full": [(n, k, "ue8m0", o, synth.M_GRID) for n, k in synth.FULL_NK for o in ("fp16", "bf16")],
    # the rowwise e4m3 GEMM (FP8_Dynamic: one scale per token and per weight
    # row), table format "rw8": the decode sweep's shapes plus two large M
    "rowwise": [(n, k, "rw8", "bf16", synth.DECODE_M + (2048, 4096)) for n, k in synth.DECODE_NK],
    # rowwise INT8 ("ri8") and block INT8 ("bi8"): both INT8 kernels compete
    # (warp-level int8 MMA, mma_scale 0; two e4m3 planes, mma_scale 1)
    "rowwise_int8": [(n, k, "ri8", "bf16", synth.DECODE_M + (2048, 4096))
                     for n, k in synth.DECODE_NK],
    "block_int8": [(n, k, "bi8", "bf16", synth.DECODE_M + (2048, 4096))
                   for n, k in synth.DECODE_NK],
}

INT8_FMTS = ("ri8", "bi8")

# grouped (MoE) GEMM, table formats "gue8m0" / "gfp32" keyed by the rows per
# expert M_max: (N, K, scale fmt, out dtype, token counts routed over E local
# experts as the MoE workload routes them)
GROUPED_SETS = {
    "moe": [(n, k, "ue8m0", "bf16", (32, 128, 512, 1024, 2048, 4096, 8192))
            for n, k in synth.MOE_NK],
}


def device_table_path() -> str:
    name = torch.cuda.get_device_name().replace(" ", "_")
    return os.path.join(HERE, "tables", f"{name}.tbl")


def candidates(M: int, N: int, K: int, fmt: str = "fp32"):
    """(kind, block_n, split, mma_scale) tuples (rw8: the rowwise kernel has
    neither the block-scaled MMA nor 64-row tiles)."""
    G = K // 128
    if fmt in INT8_FMTS:
        return int8_candidates(M, G)
    mx = fmt == "ue8m0" and K % 512 == 0
    rw = fmt == "rw8"
    out = []
    if M <= 128:
        tok = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128
        bns = sorted({tok, max(16, tok // 2)})
        for bn in bns:
            for split in (0, 1, 2, 3, 4, 6, 8):
                if split <= G:
                    out += [("swap", bn, split, m) for m in ((0, 1) if mx else (0,))]
                    if bn <= 32 and not rw:
                        out.append(("swap64", bn, split, 0))
    else:
        for bn in (128, 256):
            for split in (0, 1, 2):
                out += [("normal", bn, split, m) for m in ((0, 1) if mx else (0,))]
        for split in (0, 1):
            out += [("swap", 128, split, m) for m in ((0, 1) if mx else (0,))]
    return out


def int8_candidates(M: int, G: int):
    """INT8: the warp-level kernel (swap-AB, token tiles from 8) up to 128
    tokens, the two-plane kernel from 32 tokens (swap-AB, and normal tiles
    above 128 tokens)."""
    out = []
    splits = [sp for sp in (0, 1, 2, 3, 4, 6, 8) if sp <= G]
    if M <= 128:
        tok = 8 if M <= 8 else 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128
        for bn in sorted({tok, max(8, tok // 2)}):
            out += [("swap", bn, sp, 0) for sp in splits]
        if M >= 32:
            for bn in sorted({max(16, tok), max(16, tok // 2)}):
                out += [("swap", bn, sp, 1) for sp in (0, 1, 2) if sp <= G]
    else:
        for bn in (128, 256):
            out += [("normal", bn, sp, 1) for sp in (0, 1, 2) if sp <= G]
        out += [("swap", 128, sp, 1) for sp in (0, 1) if sp <= G]
    return out


def run_variant(aq, as_, wq, ws, v, fmt, out_dt, out, ws_buf):
    if fmt == "ri8":
        fp8bq.fp8bq_gemm_rowwise(aq, as_, wq, ws, "int8", out_dt, out=out, workspace=ws_buf,
                                 variant=v)
    elif fmt == "bi8":
        fp8bq.fp8bq_gemm_int8_block(aq, as_, wq, ws, out_dt, out=out, workspace=ws_buf,
                                    variant=v)
    elif fmt == "rw8":
        fp8bq.fp8bq_gemm_rowwise(aq, as_, wq, ws, "e4m3", out_dt, out=out, workspace=ws_buf,
                                 variant=v)
    else:
        fp8bq.fp8bq_gemm_variant(aq, as_, wq, ws, v, fmt=fmt, out_dtype=out_dt, out=out,
                                 workspace=ws_buf)


def time_variant(aq, as_, copies, ws, v, fmt, out_dt, out, ws_buf, batch=24, reps=3):
    return time_calls(lambda c: run_variant(aq, as_, c, ws, v, fmt, out_dt, out, ws_buf),
                      copies, batch, reps)


def tune_shape(N, K, fmt, out_name, Ms, log):
    dev = torch.device("cuda")
    out_dt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[out_name]
    w = torch.from_numpy(synth.weight_bf16(N, K).view(np.int16)).view(torch.bfloat16).to(dev)
    rw = fmt == "rw8"
    if fmt == "ri8":
        wq, ws = fp8bq.fp8bq_quant_rows(w, "int8")
    elif fmt == "bi8":
        wq, ws = fp8bq.fp8bq_quant_weight_int8(w)
    elif rw:
        wq, ws = fp8bq.fp8bq_quant_rows(w, "e4m3")
    else:
        wq, ws = fp8bq.fp8bq_quant_weight(w, fmt)
    del w
    n_copies = max(2, int(np.ceil(L2_BYTES / (N * K))) + 1)
    copies = [wq] + [wq.clone() for _ in range(n_copies - 1)]
    rows = []
    for M in Ms:
        x = torch.from_numpy(synth.act_decode(M, K).view(np.int16)).view(torch.bfloat16).to(dev)
        if fmt == "ri8":
            aq, as_ = fp8bq.fp8bq_quant_rows(x, "int8")
        elif fmt == "bi8":
            aq, as_ = fp8bq.fp8bq_quant_act_int8(x)
        elif rw:
            aq, as_ = fp8bq.fp8bq_quant_rows(x, "e4m3")
        else:
            aq, as_ = fp8bq.fp8bq_quant_act(x, fmt)
        out = torch.empty((M, N), dtype=out_dt, device=dev)
        results = []
        for kind, bn, split, mx in candidates(M, N, K, fmt):
            v = fp8bq.make_variant(kind, bn, split, 0, mx)
            if fmt == "ri8":
                need = fp8bq.fp8bq_rowwise_variant_workspace_bytes(M, N, K, "int8", v)
            elif fmt == "bi8":
                need = fp8bq.lib().fp8bq_int8_block_variant_workspace_bytes(M, N, K,
                                                                            ctypes.byref(v))
            elif rw:
                need = fp8bq.fp8bq_rowwise_variant_workspace_bytes(M, N, K, "e4m3", v)
            else:
                need = fp8bq.fp8bq_variant_workspace_bytes(M, N, K, v)
            if need == 0 and split != 1:
                continue  # not supported for this shape (e.g. too many tiles for tickets)
            ws_buf = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=dev)
            t = time_variant(aq, as_, copies, ws, v, fmt, out_dt, out, ws_buf)
            results.append((t, kind, bn, split, mx))
        results.sort()

        def name(r):
            return f"{r[1]}/{r[2]}/s{r[3]}" + ("/mx" if r[4] else "")

        t, kind, bn, split, mx = results[0]
        rows.append(f"{N} {K} {fmt} {out_name} {M} {kind} {bn} {split} 0 {mx}")
        best_promo = min((r for r in results if not r[4]), default=None)
        log(f"  N={N} K={K} {fmt}/{out_name} M={M}: best {name(results[0])} {t:.2f} us "
            f"(next {name(results[1])} {results[1][0]:.2f} us"
            + (f"; best promotion {name(best_promo)} {best_promo[0]:.2f} us" if best_promo else "")
            + ")" if len(results) > 1 else f"  M={M}: {name(results[0])} {t:.2f} us")
    del copies
    torch.cuda.empty_cache()
    return rows


def tune_grouped(N, K, fmt, out_name, token_counts, log):
    """Grouped entries: E = the MoE workload's local experts, counts from its
    routing; weights and activations random on the device (timing only).  One
    weight copy: every launch reads the occupied experts' weights, far more
    than the L2 holds."""
    dev = torch.device("cuda")
    E = synth.MOE_E_LOCAL
    out_dt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[out_name]
    g = torch.Generator(device=dev)
    g.manual_seed(synth.SEED_WEIGHT)
    w = torch.randn((E * N, K), device=dev, generator=g, dtype=torch.bfloat16) * 0.02
    wq, ws = fp8bq.fp8bq_quant_weight(w, fmt)
    del w
    copies = [wq, wq]
    rows, seen = [], set()
    for T in token_counts:
        counts = synth.moe_counts(E, T)
        M_max = int((counts.max() + 3) // 4 * 4)
        if M_max in seen:
            continue
        seen.add(M_max)
        cnt = torch.from_numpy(counts).to(dev)
        x = torch.randn((E * M_max, K), device=dev, generator=g, dtype=torch.bfloat16)
        aq, as_ = fp8bq.fp8bq_quant_act(x, fmt)
        del x
        out = torch.empty((E * M_max, N), dtype=out_dt, device=dev)
        results = []
        for kind, bn, split, mx in candidates(M_max, N, K, fmt):
            v = fp8bq.make_variant(kind, bn, split, 0, mx)
            need = fp8bq.fp8bq_grouped_variant_workspace_bytes(E, M_max, N, K, v)
            ws_buf = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=dev)

            def run(c, v=v, ws_buf=ws_buf):
                fp8bq.fp8bq_grouped_gemm(aq, as_, c, ws, cnt, fmt=fmt, out_dtype=out_dt, out=out,
                                         workspace=ws_buf, variant=v)
            try:
                run(wq)  # the planner rejects shapes the kernels lack, on the host
            except fp8bq.Fp8bqError:
                continue
            results.append((time_calls(run, copies), kind, bn, split, mx))
        results.sort()
        t, kind, bn, split, mx = results[0]
        rows.append(f"{N} {K} g{fmt} {out_name} {M_max} {kind} {bn} {split} 0 {mx}")
        dflt = fp8bq.fp8bq_select_grouped_variant(E, M_max, N, K, fmt, out_dt)
        log(f"  N={N} K={K} g{fmt}/{out_name} T={T} M_max={M_max}: best "
            f"{kind}/{bn}/s{split}{'/mx' if mx else ''} {t:.2f} us; "
            f"{len(results)} candidates; default {dflt['kind']}/{dflt['block_n']}/"
            f"s{dflt['split']}{'/mx' if dflt['mma_scale'] else ''}")
    del copies, wq
    torch.cuda.empty_cache()
    return rows


def time_calls(run, copies, batch=24, reps=3):
    """Best of `reps` mean launch times (us) of `batch` calls of run(copy),
    copies rotated, queued behind a GPU sleep so host time does not count."""
    for c in copies[:2]:
        run(c)
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(1_000_000)
        a.record()
        for i in range(batch):
            run(copies[i % len(copies)])
        b.record()
        b.synchronize()
        t = a.elapsed_time(b) * 1e3 / batch
        best = t if best is None else min(best, t)
    return best


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--sets", default="small,decode,prefill,full")
    ap.add_argument("--out", default=None)
    args = ap.parse_args()
    path = args.out or device_table_path()
    os.makedirs(os.path.dirname(path), exist_ok=True)
    keep = {}
    if os.path.exists(path):
        for line in open(path):
            body = line.split("#")[0].split()
            if len(body) in (9, 10):
                keep[tuple(body[:5])] = " ".join(body)
    os.environ.pop("FP8BQ_TABLE", None)
    # time without any table influence: explicit variants only
    t0 = time.time()
    done = set()
    for name in args.sets.split(","):
        if name in GROUPED_SETS:
            for (N, K, fmt, out_name, toks) in GROUPED_SETS[name]:
                print(f"tuning grouped N={N} K={K} {fmt}/{out_name} over tokens={list(toks)}",
                      flush=True)
                for row in tune_grouped(N, K, fmt, out_name, toks, lambda s: print(s, flush=True)):
                    keep[tuple(row.split()[:5])] = row
            continue
        for (N, K, fmt, out_name, Ms) in SETS[name]:
            key = (N, K, fmt, out_name)
            Ms = tuple(m for m in Ms if (key, m) not in done)
            if not Ms:
                continue
            print(f"tuning N={N} K={K} {fmt}/{out_name} over M={list(Ms)}", flush=True)
            for row in tune_shape(N, K, fmt, out_name, Ms, lambda s: print(s, flush=True)):
                f = row.split()
                keep[tuple(f[:5])] = row
            done |= {(key, m) for m in Ms}
    lines = sorted(keep.values(), key=lambda r: tuple(int(x) if x.isdigit() else x
                                                      for x in r.split()))
    with open(path, "w") as f:
        f.write("# fp8bq variant table, measured by block_scaled_fp8_group_gb300/tune.py on "
                f"{torch.cuda.get_device_name()}\n")
        f.write("# N K fmt out M kind block_n split grid mma_scale\n")
        for r in lines:
            f.write(r + "\n")
    print(f"wrote {len(lines)} entries to {path} in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
