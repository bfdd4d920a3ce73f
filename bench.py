"""Benchmark of the W8A8 block-FP8 linear hot path on GB300.

Workload (one "step"): the decode sweep -- (N, K) in {(7168, 18432),
(18432, 7168), (4096, 7168)} x M in {1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128},
33 problems; per problem the activation quant (bf16 -> e4m3 + packed UE8M0
scales) and the block-scaled GEMM (UE8M0, bf16 out) in the variant the
per-shape table selects.  Activations: bf16 N(0,1) with 1% of the K channels
x30; weights bf16 N(0,0.02) quantised 128x128 (UE8M0) once, outside the timed
region (as the pages' benchmark does).  Every GEMM of a step reads its own
copy of the weights (3.2 GB per step), so no GEMM finds its operands in L2.

Reported: value = algorithmic bytes of the whole step / step time (GB/s),
per-problem GEMM us / TFLOPS / GB/s / roofline fraction, the roofline of the
dominant kernel (the GEMM) against the measured HBM copy bandwidth, an
end-to-end number through fp8bq_linear with pinned host buffers, and the CPU
oracle timed on a bounded sample.  `--impl reference` times the oracle alone.

`--workload moe` times the grouped (mixture-of-experts) path instead: 32 local
experts of DeepSeek-V3's routed-expert projections (gate+up N=4096 K=7168,
down N=7168 K=2048), tokens routed top-8 of 256 experts with a seeded skewed
popularity, a decode batch (128 tokens) and a prefill chunk (4096 tokens);
per problem one fp8bq_grouped_linear call (quant of the occupied rows +
grouped GEMM).

`--workload rowwise --code e4m3|int8` times the per-token x per-channel
formats (FP8_Dynamic, W8A8_INT8) on the decode sweep's problems, one
fp8bq_linear_rowwise per problem, and the rowwise GEMM alone at M = 2048 and
4096 on the same (N,K).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_scaled_fp8_group_gb300 import synth  # noqa: E402

METRIC = "block-FP8 GEMM µs, TFLOPS and GB/s per (M,N,K) on 1 GB300; % of roofline"
WORKLOAD = ("decode sweep: (N,K) in {(7168,18432),(18432,7168),(4096,7168)} x "
            "M in {1,2,4,8,16,24,32,48,64,96,128}; act bf16 N(0,1), 1% channels x30 -> "
            "per-token-group quant (UE8M0 packed); weights bf16 N(0,0.02) 128x128 UE8M0; "
            "bf16 out")
# The pages' DeepGEMM numbers on H100 80GB HBM3 for shapes of this sweep
# ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §3.2, DeepGEMM table) -- context only.
H100_DEEPGEMM_US = {(8, 7168, 18432): 70.8, (8, 18432, 7168): 69.3, (8, 4096, 7168): 102.9,
                    (64, 7168, 18432): 69.4, (64, 18432, 7168): 70.4, (64, 4096, 7168): 69.1,
                    (128, 7168, 18432): 71.9, (128, 18432, 7168): 69.3,
                    (128, 4096, 7168): 141.1}
FP8_TO_BF16_NOMINAL = 2.0  # 4.5 / 2.25 PFLOP/s dense, nominal ratio


def problems():
    return [(M, N, K) for M in synth.DECODE_M for (N, K) in synth.DECODE_NK]


def gemm_bytes(M, N, K):
    """Algorithmic bytes of one GEMM launch: e4m3 A and W, packed UE8M0 act
    scales, fp32 weight scales, bf16 output."""
    G = K // 128
    Mp = (M + 3) // 4 * 4
    return M * K + N * K + 4 * Mp * ((G + 3) // 4) + 4 * ((N + 127) // 128) * G + 2 * M * N


def quant_bytes(M, K):
    G = K // 128
    Mp = (M + 3) // 4 * 4
    return 2 * M * K + M * K + 4 * Mp * ((G + 3) // 4)


def step_bytes(M, N, K):
    """Algorithmic bytes of one problem of the step (linear layer): bf16 A in,
    W, weight scales, bf16 out (the intermediate codes are not counted)."""
    G = K // 128
    return 2 * M * K + N * K + 4 * ((N + 127) // 128) * G + 2 * M * N


def gemm_flops(M, N, K):
    """The pages' TFLOPS numerator: 2*m*n*k ("vLLM DeepGEMM FP8 Block GEMM 基准测试"
    §4.3)."""
    return 2.0 * M * N * K


def pages_gbs_bytes(M, N, K):
    """The pages' GB/s numerator: m*k + k*n + 2*m*n ("vLLM DeepGEMM FP8 Block GEMM
    基准测试" §4.3)."""
    return M * K + K * N + 2 * M * N


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def variant_name(v: dict) -> str:
    """kind/block_n/s<split>, with /mx when the tensor core applies the scales."""
    return "{kind}/{block_n}/s{split}".format(**v) + ("/mx" if v.get("mma_scale") else "")


def gemm_source_hash():
    h = hashlib.sha256()
    for f in ("gemm.cu", "ptx.cuh", "internal.h"):
        h.update(open(os.path.join(ROOT, "block_scaled_fp8_group_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profile_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_decode_sweep_traffic.txt")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    t = re.search(r"traffic_bytes_per_launch_avg:\s*([0-9.eE+]+)", txt)
    if not m or not t or m.group(1) != gemm_source_hash():
        return None
    return float(t.group(1))


# ------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm_max = max(r[1] for r in rows)
        loaded = [r for r in rows if r[0] > 0.5 * sm_max] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[2]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in loaded])), "sm_max_mhz": sm_max,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded)}


# ------------------------------------------------------------- oracle legs

_ORACLE_W = {}


def oracle_time_sample(rows_per_shape=1, reps=1):
    """Times the CPU oracle (quant of the sampled rows + their GEMM rows) on
    one thread; returns (extrapolated whole-step seconds, sample seconds,
    description).  Weights are quantised by the oracle outside the timing."""
    import oracle
    total_rows = sum(synth.DECODE_M)
    est = 0.0
    sample_s = 0.0
    for (N, K) in synth.DECODE_NK:
        if (N, K) not in _ORACLE_W:
            _ORACLE_W[(N, K)] = oracle.quant_weight(synth.weight_bf16(N, K), oracle.BF16, 128,
                                                    128, True)
        qw, sw = _ORACLE_W[(N, K)]
        xb = synth.act_decode(rows_per_shape, K)
        best = None
        for _ in range(reps):
            t0 = time.perf_counter()
            qa, sa = oracle.quant_act(xb, oracle.BF16, 128, True)
            oracle.gemm(qa, sa, qw, sw, True)
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        sample_s += best
        est += best / rows_per_shape * total_rows
    desc = (f"{rows_per_shape} activation row(s) per (N,K) through oracle quant + fp64 GEMM "
            f"(all N columns), single thread; whole-step time extrapolated linearly in M "
            f"({total_rows} rows per (N,K))")
    return est, sample_s, desc


def oracle_time_all_cores(threads=None):
    """The same oracle routine over row partitions on all host cores: one row
    per thread per (N,K), quant + fp64 GEMM row, threads around the unchanged
    single-thread C calls (ctypes releases the GIL).  Returns (extrapolated
    whole-step seconds, threads, description)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    n = threads or os.cpu_count() or 1
    total_rows = sum(synth.DECODE_M)
    est = 0.0
    for (N, K) in synth.DECODE_NK:
        if (N, K) not in _ORACLE_W:
            _ORACLE_W[(N, K)] = oracle.quant_weight(synth.weight_bf16(N, K), oracle.BF16, 128,
                                                    128, True)
        qw, sw = _ORACLE_W[(N, K)]
        xb = synth.act_decode(n, K)

        def one(r):
            qa, sa = oracle.quant_act(np.ascontiguousarray(xb[r:r + 1]), oracle.BF16, 128, True)
            oracle.gemm(qa, sa, qw, sw, True)

        with ThreadPoolExecutor(max_workers=n) as ex:
            t0 = time.perf_counter()
            list(ex.map(one, range(n)))
            dt = time.perf_counter() - t0
        est += dt / n * total_rows
    desc = (f"{n} activation rows per (N,K), one per thread on {n} threads (row partitions of "
            "the same single-thread oracle routine); extrapolated linearly in M")
    return est, n, desc


def max_over_ranks(seconds: float, device) -> float:
    """The slowest rank's time: replicas report the whole job's throughput as
    the units all ranks processed over the time of the slowest one."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job GB/s of `world` replicas that each moved bytes_per_rank in
    `seconds` (the max over ranks): weak scaling."""
    return world * bytes_per_rank / seconds / 1e9


def total_step_bytes():
    return sum(step_bytes(M, N, K) for (M, N, K) in problems())


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    steps, warm = args.steps_ref, max(0, args.warmup)
    for _ in range(warm):
        oracle_time_sample(1)
    ests = []
    t0 = time.perf_counter()
    for _ in range(steps):
        est, _, desc = oracle_time_sample(1)
        ests.append(est)
    wall = time.perf_counter() - t0
    est = float(np.mean(ests))
    value = total_step_bytes() / est / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": est * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- MoE workload

MOE_WORKLOAD = ("moe: 32 local experts, DeepSeek-V3 routed-expert projections (N,K) in "
                "{(4096,7168),(7168,2048)}; tokens {128, 4096} routed top-8 of 256 experts "
                "(seeded Dirichlet(0.5) popularity), rows per expert padded to the largest "
                "count (multiple of 4); act bf16 N(0,1) 1% channels x30; weights bf16 "
                "N(0,0.02) 128x128 UE8M0; bf16 out; fp8bq_grouped_linear per problem")


def moe_problems():
    """(tokens, N, K, counts, M_max) of the MoE step."""
    out = []
    for T in synth.MOE_TOKENS:
        counts = synth.moe_counts(synth.MOE_E_LOCAL, T)
        M_max = int((counts.max() + 3) // 4 * 4)
        for (N, K) in synth.MOE_NK:
            out.append((T, N, K, counts, M_max))
    return out


def moe_bytes(N, K, counts, linear):
    """Algorithmic bytes of one grouped problem: the weights and weight scales
    of the experts that hold tokens, and the occupied rows (bf16 in for the
    linear layer; e4m3 codes + packed scales for the GEMM alone), bf16 out."""
    G = K // 128
    ne = int((counts > 0).sum())
    toks = int(counts.sum())
    w = ne * (N * K + 4 * (N // 128) * G)
    a = 2 * toks * K if linear else toks * K + 4 * ((G + 3) // 4) * toks
    return w + a + 2 * toks * N


def run_gpu_moe(args, rank, world):
    import torch
    import torch.distributed as dist

    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    E = synth.MOE_E_LOCAL
    probs = moe_problems()
    wq, ws, xs, cnts, outs, variants = [], [], [], [], [], []
    w_cache = {}
    for (T, N, K, counts, M_max) in probs:
        if (N, K) not in w_cache:
            q = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
            s = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=dev)
            wb = synth.moe_weight_bf16(E, N, K)
            for e in range(E):
                wd = torch.from_numpy(wb[e].view(np.int16)).view(torch.bfloat16).to(dev)
                fp8bq.fp8bq_quant_weight(wd, "ue8m0", q=q[e], s=s[e])
            del wb
            w_cache[(N, K)] = (q, s)
        q, s = w_cache[(N, K)]
        wq.append(q.clone())  # every problem reads its own copy (> L2 each)
        ws.append(s)
        xb = synth.moe_act(E, M_max, K)
        xs.append(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev))
        cnts.append(torch.from_numpy(counts).to(dev))
        outs.append(torch.empty((E * M_max, N), dtype=torch.bfloat16, device=dev))
        variants.append(fp8bq.fp8bq_select_grouped_variant(E, M_max, N, K, "ue8m0"))
    del w_cache
    ws_bytes = max(fp8bq.fp8bq_grouped_linear_workspace_bytes(E, p[4], p[1], p[2], "ue8m0")
                   for p in probs)
    wspace = torch.zeros(ws_bytes + (1 << 20), dtype=torch.uint8, device=dev)
    aqs = [torch.empty((E * p[4], p[2]), dtype=torch.uint8, device=dev) for p in probs]
    ass = [torch.empty(fp8bq.act_scale_shape(E * p[4], p[2], 128, "ue8m0")[0],
                       dtype=torch.int32, device=dev) for p in probs]
    gws = torch.zeros(max(fp8bq.fp8bq_grouped_gemm_workspace_bytes(E, p[4], p[1], p[2], "ue8m0")
                          for p in probs) + (1 << 20), dtype=torch.uint8, device=dev)

    def step():
        for i in range(len(probs)):
            fp8bq.fp8bq_grouped_linear(xs[i], wq[i], ws[i], cnts[i], fmt="ue8m0", out=outs[i],
                                       workspace=wspace)

    mk = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in probs]
    ev_s, ev_e, ev2_s, ev2_e = mk(), mk(), mk(), mk()

    def step_split():
        for i in range(len(probs)):
            fp8bq.fp8bq_quant_act(xs[i], "ue8m0", q=aqs[i], s=ass[i])
            ev[i][0].record()
            fp8bq.fp8bq_grouped_gemm(aqs[i], ass[i], wq[i], ws[i], cnts[i], fmt="ue8m0",
                                     out=outs[i], workspace=gws)
            ev[i][1].record()

    step()
    step_split()
    torch.cuda.synchronize()
    g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g1, stream=side):
            ev_s.record()
            step()
            ev_e.record()
        with torch.cuda.graph(g2, stream=side):
            ev2_s.record()
            step_split()
            ev2_e.record()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        g1.replay()
        g2.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    step_ms = []
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        g1.replay()
        ev_e.synchronize()
        step_ms.append(ev_s.elapsed_time(ev_e))
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    step_s = float(np.mean(step_ms)) / 1e3
    n_instr = max(1, min(args.steps, args.instr_steps))
    gemm_ms = np.zeros(len(probs))
    for _ in range(n_instr):
        g2.replay()
        ev2_e.synchronize()
        gemm_ms += np.array([a.elapsed_time(b) for a, b in ev])
    gemm_us = gemm_ms / n_instr * 1e3
    assert fp8bq.fp8bq_device_status() == 0

    # end to end: activations and counts from pinned host memory, outputs back
    hx = [x.cpu().pin_memory() for x in xs]
    hc = [c.cpu().pin_memory() for c in cnts]
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    h2d = sum(x.numel() * 2 + c.numel() * 4 for x, c in zip(hx, hc))
    d2h = sum(o.numel() * 2 for o in ho)

    def e2e_step():
        for i in range(len(probs)):
            xs[i].copy_(hx[i], non_blocking=True)
            cnts[i].copy_(hc[i], non_blocking=True)
            fp8bq.fp8bq_grouped_linear(xs[i], wq[i], ws[i], cnts[i], fmt="ue8m0", out=outs[i],
                                       workspace=wspace)
            ho[i].copy_(outs[i], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    g3 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g3, stream=side):
            e2e_step()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        g3.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(1, min(args.steps, args.e2e_steps))
    a.record()
    for _ in range(n_e2e):
        g3.replay()
    b.record()
    b.synchronize()
    e2e_s = a.elapsed_time(b) / 1e3 / n_e2e
    step_total = sum(moe_bytes(p[1], p[2], p[3], True) for p in probs)
    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_TO_BF16_NOMINAL
    per = []
    for i, (T, N, K, counts, M_max) in enumerate(probs):
        t = gemm_us[i] * 1e-6
        byt = moe_bytes(N, K, counts, False)
        fl = 2.0 * int(counts.sum()) * N * K
        t_roof = max(byt / (peaks["hbm_gbs"] * 1e9), fl / (fp8_peak * 1e12))
        per.append({"tokens": T, "n": N, "k": K, "experts": E, "m_max": M_max,
                    "experts_with_tokens": int((counts > 0).sum()),
                    "token_rows": int(counts.sum()), "us": round(gemm_us[i], 3),
                    "tflops": round(fl / t / 1e12, 2), "gbs_alg": round(byt / t / 1e9, 1),
                    "roofline_frac": round(t_roof / t, 3),
                    "variant": variant_name(variants[i])})
    tot_gemm = sum(moe_bytes(p[1], p[2], p[3], False) for p in probs)
    achieved = tot_gemm / (gemm_us.sum() * 1e-6) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        est, sample_s, desc = moe_oracle_sample()
        cpu = {"value": step_total / est / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": desc + f" (sample took {sample_s:.1f} s)"}
    line = {
        "metric": METRIC, "value": round(step_total / step_s / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": MOE_WORKLOAD, "problems_per_step": len(probs),
                   "l2": "inputs larger than L2: every problem reads its own weight copy "
                         "(0.47-0.94 GB each)",
                   "timing": "graph: step = fp8bq_grouped_linear per problem, CUDA events on "
                             "the launching stream; per-GEMM durations from an instrumented "
                             "pass (quant and grouped GEMM as separate calls)",
                   "parallelism": "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": None,
                     "kernel": "grouped block-FP8 GEMM (gemm_kernel / gemm_mx_kernel, grouped "
                               "tiles), 4 launches per step",
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy)"},
        "cpu_baseline": cpu,
        "e2e": {"value": step_total / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3, "steps": n_e2e,
                "api": "fp8bq_grouped_linear per problem (graph), activations and counts "
                       "copied in from pinned host memory and outputs copied back each step"},
        "gpu_launches": args.steps * 2 * len(probs), "clocks": clk, "per_shape": per,
        "wall_timed_s": round(t_wall, 3), "gemm_source_sha256_16": gemm_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


def moe_oracle_sample():
    """The oracle on one thread over one token row of each MoE problem (quant
    of the row + its GEMM row against its expert's weights), extrapolated
    linearly to the problem's token rows."""
    import oracle
    est, sample_s = 0.0, 0.0
    for (T, N, K, counts, M_max) in moe_problems():
        e = int(np.argmax(counts > 0))
        wb = synth.moe_weight_bf16(1, N, K, seed=synth.SEED_WEIGHT + 1000 * e)[0]
        qw, sw = oracle.quant_weight(wb, oracle.BF16, 128, 128, True)
        xb = synth.act_decode(1, K)
        t0 = time.perf_counter()
        qa, sa = oracle.quant_act(xb, oracle.BF16, 128, True)
        oracle.gemm(qa, sa, qw, sw, True)
        dt = time.perf_counter() - t0
        sample_s += dt
        est += dt * int(counts.sum())
    return est, sample_s, ("one token row per MoE problem through oracle quant + fp64 GEMM "
                           "(all N columns of its expert), single thread; extrapolated "
                           "linearly to each problem's token rows")


# ----------------------------------------------- rowwise (per-token x per-channel)

ROWWISE_WORKLOAD = ("{code}: decode sweep (N,K) in {{(7168,18432),(18432,7168),(4096,7168)}} "
                    "x M in {{1,2,4,8,16,24,32,48,64,96,128}}; act bf16 N(0,1), 1% channels x30 "
                    "-> {aq}; weights bf16 N(0,0.02) {wq}; bf16 out; {api} per problem")
ROWWISE_QUANT = {"e4m3": ("per-token quant", "per-channel quant", "fp8bq_linear_rowwise"),
                 "int8": ("per-token quant", "per-channel quant", "fp8bq_linear_rowwise"),
                 "int8block": ("1x128 group quant", "128x128 block quant",
                               "fp8bq_linear_int8_block")}
ROWWISE_PREFILL_M = (2048, 4096)


def rowwise_gemm_bytes(M, N, K):
    """Algorithmic bytes of one rowwise GEMM: codes of A and W (1 byte each),
    one fp32 scale per token and per weight row, bf16 output."""
    return M * K + N * K + 4 * M + 4 * N + 2 * M * N


def rowwise_step_bytes(M, N, K):
    return 2 * M * K + N * K + 4 * N + 2 * M * N


def block_int8_gemm_bytes(M, N, K):
    """Block INT8 GEMM: int8 codes, fp32 act scales [G][Mp], fp32 weight
    block scales, bf16 out."""
    G, Mp = K // 128, (M + 3) // 4 * 4
    return M * K + N * K + 4 * Mp * G + 4 * ((N + 127) // 128) * G + 2 * M * N


def block_int8_step_bytes(M, N, K):
    G = K // 128
    return 2 * M * K + N * K + 4 * ((N + 127) // 128) * G + 2 * M * N


class FormatCalls:
    """The calls one per-token x per-channel code (e4m3, int8) or block INT8
    (int8block) makes, so one benchmark leg serves all three."""

    def __init__(self, fp8bq, torch, code):
        self.f, self.t, self.code = fp8bq, torch, code
        self.block = code == "int8block"

    def quant_w(self, wd):
        if self.block:
            return self.f.fp8bq_quant_weight_int8(wd)
        return self.f.fp8bq_quant_rows(wd, self.code)

    def alloc_a(self, M, K, dev):
        t = self.t
        qdt = t.int8 if self.code != "e4m3" else t.uint8
        if self.block:
            shape = self.f.act_scale_shape(M, K, 128, "fp32")[0]
            return t.empty((M, K), dtype=qdt, device=dev), t.empty(shape, dtype=t.float32,
                                                                     device=dev)
        return t.empty((M, K), dtype=qdt, device=dev), t.empty(M, dtype=t.float32, device=dev)

    def quant_a(self, x, q=None, s=None):
        if self.block:
            return self.f.fp8bq_quant_act_int8(x, q=q, s=s)
        return self.f.fp8bq_quant_rows(x, self.code, q=q, s=s)

    def gemm(self, aq, as_, wq, ws, out, workspace):
        if self.block:
            return self.f.fp8bq_gemm_int8_block(aq, as_, wq, ws, self.t.bfloat16, out=out,
                                                workspace=workspace)
        return self.f.fp8bq_gemm_rowwise(aq, as_, wq, ws, self.code, self.t.bfloat16, out=out,
                                         workspace=workspace)

    def linear(self, x, wq, ws, out, workspace):
        if self.block:
            return self.f.fp8bq_linear_int8_block(x, wq, ws, self.t.bfloat16, out=out,
                                                  workspace=workspace)
        return self.f.fp8bq_linear_rowwise(x, wq, ws, self.code, self.t.bfloat16, out=out,
                                           workspace=workspace)

    def linear_ws(self, M, N, K):
        if self.block:
            return self.f.lib().fp8bq_linear_int8_block_workspace_bytes(M, N, K, 0)
        return self.f.fp8bq_linear_rowwise_workspace_bytes(M, N, K, self.code, self.t.bfloat16)

    def gemm_ws(self, M, N, K):
        if self.block:
            return self.f.lib().fp8bq_int8_block_workspace_bytes(M, N, K, 0)
        return self.f.fp8bq_rowwise_workspace_bytes(M, N, K, self.code, self.t.bfloat16)

    def select(self, M, N, K):
        if self.block:
            return self.f.fp8bq_select_int8_block_variant(M, N, K, self.t.bfloat16)
        return self.f.fp8bq_select_rowwise_variant(M, N, K, self.code, self.t.bfloat16)

    def gemm_bytes(self, M, N, K):
        return block_int8_gemm_bytes(M, N, K) if self.block else rowwise_gemm_bytes(M, N, K)

    def step_bytes(self, M, N, K):
        return block_int8_step_bytes(M, N, K) if self.block else rowwise_step_bytes(M, N, K)


def run_gpu_rowwise(args, rank, world):
    import torch

    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq

    code = args.code
    fc = FormatCalls(fp8bq, torch, code)
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    probs = problems()
    w_q, w_s = {}, {}
    for (N, K) in synth.DECODE_NK:
        wd = torch.from_numpy(synth.weight_bf16(N, K).view(np.int16)).view(torch.bfloat16).to(dev)
        q, s = fc.quant_w(wd)
        del wd
        for M in synth.DECODE_M:
            w_q[(M, N, K)] = q.clone()  # every problem reads its own weight copy (> L2 in total)
        w_s[(N, K)] = s
        del q
    xs, aqs, ass, outs = {}, {}, {}, {}
    for p in probs:
        M, N, K = p
        xs[p] = torch.from_numpy(synth.act_decode(M, K).view(np.int16)).view(torch.bfloat16).to(dev)
        aqs[p], ass[p] = fc.alloc_a(M, K, dev)
        outs[p] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws_bytes = max(fc.linear_ws(*p) for p in probs)
    ws = torch.zeros(ws_bytes + (1 << 20), dtype=torch.uint8, device=dev)
    variants = {p: fc.select(*p) for p in probs}
    mk = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in probs]
    ev_s, ev_e, ev2_s, ev2_e = mk(), mk(), mk(), mk()

    def step():
        for p in probs:
            fc.linear(xs[p], w_q[p], w_s[(p[1], p[2])], outs[p], ws)

    def step_split():
        for i, p in enumerate(probs):
            fc.quant_a(xs[p], q=aqs[p], s=ass[p])
            ev[i][0].record()
            fc.gemm(aqs[p], ass[p], w_q[p], w_s[(p[1], p[2])], outs[p], ws)
            ev[i][1].record()

    step()
    step_split()
    torch.cuda.synchronize()
    g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g1, stream=side):
            ev_s.record()
            step()
            ev_e.record()
        with torch.cuda.graph(g2, stream=side):
            ev2_s.record()
            step_split()
            ev2_e.record()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        g1.replay()
        g2.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    step_ms = []
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        g1.replay()
        ev_e.synchronize()
        step_ms.append(ev_s.elapsed_time(ev_e))
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    step_s = float(np.mean(step_ms)) / 1e3
    n_instr = max(1, min(args.steps, args.instr_steps))
    gemm_ms = np.zeros(len(probs))
    for _ in range(n_instr):
        g2.replay()
        ev2_e.synchronize()
        gemm_ms += np.array([a.elapsed_time(b) for a, b in ev])
    gemm_us = gemm_ms / n_instr * 1e3
    assert fp8bq.fp8bq_device_status() == 0

    # large M: the GEMM alone, two weight copies alternating (each > L2 / 2)
    prefill = []
    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_TO_BF16_NOMINAL
    for (N, K) in synth.DECODE_NK:
        wq2 = [w_q[(1, N, K)], w_q[(2, N, K)]]
        for M in ROWWISE_PREFILL_M:
            xa = torch.from_numpy(synth.act_prefill(M, K).view(np.int16)).view(
                torch.bfloat16).to(dev)
            aq, as_ = fc.quant_a(xa)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsz = fc.gemm_ws(M, N, K)
            wsp = ws if wsz <= ws.numel() else torch.zeros(wsz, dtype=torch.uint8, device=dev)
            for i in range(3):
                fc.gemm(aq, as_, wq2[i % 2], w_s[(N, K)], o, wsp)
            reps = 10
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for i in range(reps):
                evs[i][0].record()
                fc.gemm(aq, as_, wq2[i % 2], w_s[(N, K)], o, wsp)
                evs[i][1].record()
            torch.cuda.synchronize()
            us = float(np.median([a.elapsed_time(b) for a, b in evs])) * 1e3
            fl = gemm_flops(M, N, K)
            entry = {"m": M, "n": N, "k": K, "us": round(us, 2),
                     "tflops": round(fl / us / 1e6, 1),
                     "variant": variant_name(fc.select(M, N, K))}
            if code == "e4m3":
                entry["frac_of_fp8_peak"] = round(fl / us / 1e6 / fp8_peak, 3)
            prefill.append(entry)
            del xa, aq, as_, o
    assert fp8bq.fp8bq_device_status() == 0

    per = []
    for i, (M, N, K) in enumerate(probs):
        t = gemm_us[i] * 1e-6
        b = fc.gemm_bytes(M, N, K)
        per.append({"m": M, "n": N, "k": K, "us": round(gemm_us[i], 3),
                    "tflops": round(gemm_flops(M, N, K) / t / 1e12, 2),
                    "gbs_alg": round(b / t / 1e9, 1),
                    "roofline_frac": round(b / (peaks["hbm_gbs"] * 1e9) / t, 3),
                    "variant": variant_name(variants[(M, N, K)])})
    tot = sum(fc.gemm_bytes(*p) for p in probs)
    achieved = tot / (gemm_us.sum() * 1e-6) / 1e9
    step_total = sum(fc.step_bytes(*p) for p in probs)
    kern = {"e4m3": "gemm_mx_kernel (rowwise: plain kind::f8f6f4, scales in the epilogue)",
            "int8": "gemm_i8_kernel (mma.sync m16n8k32 s8, TMA-fed) or gemm_mx_kernel on two "
                    "e4m3 planes, per shape from the measured table",
            "int8block": "gemm_i8_kernel (block promotion per K slab, mma.sync m16n8k32 s8) or "
                         "gemm_mx_kernel on two e4m3 planes, per shape from the measured table"}[code]
    line = {
        "metric": METRIC, "value": round(step_total / step_s / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": code, "data": "synthetic",
        "config": {"workload": ROWWISE_WORKLOAD.format(
                       code=code, aq=ROWWISE_QUANT[code][0], wq=ROWWISE_QUANT[code][1],
                       api=ROWWISE_QUANT[code][2]),
                   "problems_per_step": len(probs),
                   "l2": "inputs larger than L2: each GEMM reads its own weight copy",
                   "timing": "graph: step = fp8bq_linear_rowwise per problem, CUDA events on "
                             "the launching stream; per-GEMM durations from an instrumented "
                             "pass (quant and GEMM as separate calls)",
                   "parallelism": "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": None, "kernel": kern,
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy)"},
        "cpu_baseline": None, "e2e": None, "gpu_launches": args.steps * 2 * len(probs),
        "clocks": clk, "per_shape": per, "prefill_gemm": prefill,
        "wall_timed_s": round(t_wall, 3), "gemm_source_sha256_16": gemm_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world):
    import torch
    import torch.distributed as dist

    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    probs = problems()
    stream = torch.cuda.current_stream()

    # ---- setup (untimed): weights quantised once, one copy per M point
    w_q, w_s = {}, {}
    for (N, K) in synth.DECODE_NK:
        wb = synth.weight_bf16(N, K)
        wd = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).to(dev)
        q, s = fp8bq.fp8bq_quant_weight(wd, "ue8m0")
        del wd
        for M in synth.DECODE_M:
            w_q[(M, N, K)] = q.clone()
        w_s[(N, K)] = s
        del q
    torch.cuda.synchronize()
    xs, aqs, ass, outs = {}, {}, {}, {}
    for (M, N, K) in probs:
        xb = synth.act_decode(M, K)
        xs[(M, N, K)] = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
        aqs[(M, N, K)], ass[(M, N, K)] = (
            torch.empty((M, K), dtype=torch.uint8, device=dev),
            torch.empty(fp8bq.act_scale_shape(M, K, 128, "ue8m0")[0], dtype=torch.int32,
                        device=dev))
        outs[(M, N, K)] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws_bytes = max(fp8bq.fp8bq_linear_workspace_bytes(M, N, K, "ue8m0", torch.bfloat16)
                   for (M, N, K) in probs)
    ws = torch.zeros(ws_bytes + (1 << 20), dtype=torch.uint8, device=dev)
    variants = {p: fp8bq.fp8bq_select_variant(*p, "ue8m0", torch.bfloat16) for p in probs}

    def step_linear():
        # the timed step: one fp8bq_linear call (quant + GEMM, PDL) per problem
        for p in probs:
            M, N, K = p
            fp8bq.fp8bq_linear(xs[p], w_q[p], w_s[(N, K)], fmt="ue8m0",
                               out_dtype=torch.bfloat16, out=outs[p], workspace=ws)

    def step_split(ev_pairs):
        # the instrumented step: quant and GEMM as separate calls, with timing
        # events around every GEMM launch
        for i, p in enumerate(probs):
            M, N, K = p
            fp8bq.fp8bq_quant_act(xs[p], "ue8m0", q=aqs[p], s=ass[p])
            ev_pairs[i][0].record()
            fp8bq.fp8bq_gemm(aqs[p], ass[p], w_q[p], w_s[(N, K)], fmt="ue8m0",
                             out_dtype=torch.bfloat16, out=outs[p], workspace=ws)
            ev_pairs[i][1].record()

    def step_gemms():
        # the 33 GEMMs alone, launched back to back as in the step (PDL
        # between them), on the codes the instrumented pass wrote
        for p in probs:
            M, N, K = p
            fp8bq.fp8bq_gemm(aqs[p], ass[p], w_q[p], w_s[(N, K)], fmt="ue8m0",
                             out_dtype=torch.bfloat16, out=outs[p], workspace=ws)

    # ---- timing instruments: CUDA graphs with external timing events, else eager
    mode = args.mode
    ext_ok = True
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        ext_ok = False
    if mode == "graph" and not ext_ok:
        mode = "eager"
    mk = (lambda: torch.cuda.Event(enable_timing=True, external=True)) if mode == "graph" else \
        (lambda: torch.cuda.Event(enable_timing=True))
    ev_pairs = [(mk(), mk()) for _ in probs]
    ev_start, ev_end = mk(), mk()
    ev2_start, ev2_end = mk(), mk()
    ev3_start, ev3_end = mk(), mk()

    # first launches: load the table, set kernel attributes
    step_linear()
    step_split(ev_pairs)
    torch.cuda.synchronize()
    graphs = None
    if mode == "graph":
        g_lin, g_split, g_gemm = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g_lin, stream=side):
                ev_start.record()
                step_linear()
                ev_end.record()
            with torch.cuda.graph(g_split, stream=side):
                ev2_start.record()
                step_split(ev_pairs)
                ev2_end.record()
            with torch.cuda.graph(g_gemm, stream=side):
                ev3_start.record()
                step_gemms()
                ev3_end.record()
        torch.cuda.synchronize()
        graphs = (g_lin, g_split, g_gemm)

    def run_timed():
        if graphs is not None:
            graphs[0].replay()
        else:
            ev_start.record()
            step_linear()
            ev_end.record()

    def run_instr():
        if graphs is not None:
            graphs[1].replay()
        else:
            ev2_start.record()
            step_split(ev_pairs)
            ev2_end.record()

    def run_gemms():
        if graphs is not None:
            graphs[2].replay()
        else:
            ev3_start.record()
            step_gemms()
            ev3_end.record()

    for _ in range(args.warmup):
        run_timed()
        run_instr()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    step_ms = []
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        run_timed()
        ev_end.synchronize()
        step_ms.append(ev_start.elapsed_time(ev_end))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop() if rank == 0 else None
    step_s = float(np.mean(step_ms)) / 1e3
    if world > 1:
        step_s = max_over_ranks(step_s, dev)
    # instrumented pass (same problems, same cold weights): per-GEMM durations
    n_instr = max(1, min(args.steps, args.instr_steps))
    gemm_ms, split_ms = np.zeros(len(probs)), []
    for _ in range(n_instr):
        run_instr()
        ev2_end.synchronize()
        split_ms.append(ev2_start.elapsed_time(ev2_end))
        gemm_ms += np.array([a.elapsed_time(b) for a, b in ev_pairs])
    gemm_us = gemm_ms / n_instr * 1e3
    # the GEMM launches as the step runs them: back to back, PDL between them
    chain_ms = []
    for _ in range(n_instr):
        run_gemms()
        ev3_end.synchronize()
        chain_ms.append(ev3_start.elapsed_time(ev3_end))
    chain_s = float(np.mean(chain_ms)) / 1e3
    assert fp8bq.fp8bq_device_status() == 0
    launches = args.steps * 2 * len(probs)

    # ---- end to end through the public fp8bq_linear call with host buffers
    e2e = None
    if not args.no_e2e:
        # all inputs of a step in one pinned host buffer and all outputs in
        # another, one slice per problem (16-byte aligned: M*K and M*N are
        # multiples of 64 elements)
        x_off, o_off, xo, oo = {}, {}, 0, 0
        for (M, N, K) in probs:
            x_off[(M, N, K)], o_off[(M, N, K)] = xo, oo
            xo += M * K
            oo += M * N
        hx_all = torch.empty(xo, dtype=torch.bfloat16).pin_memory()
        hout_all = torch.empty(oo, dtype=torch.bfloat16).pin_memory()
        for (M, N, K) in probs:
            hx_all[x_off[(M, N, K)]:x_off[(M, N, K)] + M * K].copy_(xs[(M, N, K)].reshape(-1).cpu())
        xd_all = torch.empty(xo, dtype=torch.bfloat16, device=dev)
        od_all = torch.empty(oo, dtype=torch.bfloat16, device=dev)
        xd = {p: xd_all[x_off[p]:x_off[p] + p[0] * p[2]].view(p[0], p[2]) for p in probs}
        od = {p: od_all[o_off[p]:o_off[p] + p[0] * p[1]].view(p[0], p[1]) for p in probs}
        h2d, d2h = 2 * xo, 2 * oo

        hx = {p: hx_all[x_off[p]:x_off[p] + p[0] * p[2]].view(p[0], p[2]) for p in probs}
        ho = {p: hout_all[o_off[p]:o_off[p] + p[0] * p[1]].view(p[0], p[1]) for p in probs}
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

        wait_every = 6  # measured on GB300: 1 -> 3152, 6 -> 3379, 33 -> 2886 GB/s

        def e2e_step():
            # copies overlap the compute: every problem's input goes up on
            # one side stream ahead of its linear layer, and its output comes
            # back on another while the next problems run.  The compute
            # stream waits once per `wait_every` problems (for the inputs of
            # the next ones): each cross-stream wait cuts the chain of
            # programmatic launches between consecutive layers
            cur = torch.cuda.current_stream()
            h2d_s.wait_stream(cur)
            d2h_s.wait_stream(cur)
            ready = []
            with torch.cuda.stream(h2d_s):
                for p in probs:
                    xd[p].copy_(hx[p], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(h2d_s)
                    ready.append(e)
            for i, p in enumerate(probs):
                M, N, K = p
                if i % wait_every == 0:
                    cur.wait_event(ready[min(i + wait_every, len(probs)) - 1])
                fp8bq.fp8bq_linear(xd[p], w_q[p], w_s[(N, K)], fmt="ue8m0",
                                   out_dtype=torch.bfloat16, out=od[p], workspace=ws)
                done = torch.cuda.Event()
                done.record(cur)
                d2h_s.wait_event(done)
                with torch.cuda.stream(d2h_s):
                    ho[p].copy_(od[p], non_blocking=True)
            cur.wait_stream(h2d_s)
            cur.wait_stream(d2h_s)

        e2e_step()
        torch.cuda.synchronize()
        g_e2e = None
        if mode == "graph":
            g_e2e = torch.cuda.CUDAGraph()
            side2 = torch.cuda.Stream()
            side2.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side2):
                with torch.cuda.graph(g_e2e, stream=side2):
                    e2e_step()
            torch.cuda.synchronize()
        run_e2e = g_e2e.replay if g_e2e is not None else e2e_step
        for _ in range(args.warmup):
            run_e2e()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, min(args.steps, args.e2e_steps))
        a.record()
        for _ in range(n_e2e):
            run_e2e()
        b.record()
        b.synchronize()
        e2e_s = a.elapsed_time(b) / 1e3 / n_e2e
        if world > 1:
            e2e_s = max_over_ranks(e2e_s, dev)
        e2e = {"value": job_value(total_step_bytes(), world, e2e_s), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_s * 1e3, "steps": n_e2e,
               "api": f"fp8bq_linear (quant + GEMM, PDL) per problem ({mode}); every step copies "
                      "each problem's input from pinned host memory on a side stream ahead of its "
                      "linear layer (the compute waits once per 6 problems) and its output back on "
                      "another side stream after it, overlapping the compute of the other problems"}

    if rank != 0:
        return 0

    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_TO_BF16_NOMINAL
    per = []
    for i, (M, N, K) in enumerate(probs):
        t = gemm_us[i] * 1e-6
        b = gemm_bytes(M, N, K)
        fl = gemm_flops(M, N, K)
        t_roof = max(b / (peaks["hbm_gbs"] * 1e9), fl / (fp8_peak * 1e12))
        per.append({"m": M, "n": N, "k": K, "us": round(gemm_us[i], 3),
                    "tflops": round(fl / t / 1e12, 2),
                    "gbs_pages": round(pages_gbs_bytes(M, N, K) / t / 1e9, 1),
                    "gbs_alg": round(b / t / 1e9, 1), "roofline_frac": round(t_roof / t, 3),
                    "variant": variant_name(variants[(M, N, K)]),
                    "h100_deepgemm_us": H100_DEEPGEMM_US.get((M, N, K))})
    n_mx = sum(1 for p in probs if variants[p]["mma_scale"])
    tot_gemm_bytes = sum(gemm_bytes(*p) for p in probs)
    achieved = tot_gemm_bytes / chain_s / 1e9
    achieved_iso = tot_gemm_bytes / (gemm_us.sum() * 1e-6) / 1e9
    traffic = profile_traffic()
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic,
            "method": "achieved = the 33 GEMMs' algorithmic bytes / the average time of the 33 "
                      "GEMM launches run back to back as the step launches them (PDL between "
                      "them; CUDA events around the chain on the launching stream); "
                      "achieved_isolated = the same bytes / the sum of the GEMMs timed one by "
                      "one between events (each pays its own launch, ramp and tail)",
            "achieved_isolated": round(achieved_iso, 1),
            "frac_isolated": round(achieved_iso / peaks["hbm_gbs"], 4),
            "gemm_chain_ms": round(chain_s * 1e3, 4),
            "kernel": f"block-scaled FP8 GEMM, decode sweep: {len(probs)} launches per step "
                      f"({n_mx} gemm_mx_kernel, {len(probs) - n_mx} gemm_kernel, as the "
                      "table selects)",
            "algorithmic_bytes_per_launch_avg": tot_gemm_bytes / len(probs),
            "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy)"}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        est, sample_s, desc = oracle_time_sample(rows_per_shape=args.oracle_rows)
        cpu = {"value": total_step_bytes() / est / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": desc + f" (sample took {sample_s:.1f} s)"}
        est_all, nthr, desc_all = oracle_time_all_cores()
        cpu["all_cores"] = {"value": total_step_bytes() / est_all / 1e9, "unit": "GB/s",
                            "cores": nthr, "sample": desc_all}
    value = job_value(total_step_bytes(), world, step_s)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "problems_per_step": len(probs),
                   "l2": "inputs larger than L2: each GEMM reads its own weight copy "
                         "(3.2 GB of weights per step)",
                   "timing": f"{mode}: step = fp8bq_linear per problem (PDL between "
                             "kernels), CUDA events on the launching stream around each step; "
                             "per-GEMM durations (per_shape) from an instrumented pass of the "
                             "same step (quant and GEMM as separate calls, events around every "
                             "GEMM); the roofline from the same GEMMs launched back to back",
                   "instrumented_step_ms": round(float(np.mean(split_ms)), 4),
                   "instrumented_steps": n_instr,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clk, "per_shape": per, "wall_timed_s": round(t_wall, 3),
        "gemm_source_sha256_16": gemm_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("fp8bq", "reference"), default="fp8bq")
    ap.add_argument("--mode", choices=("graph", "eager"), default="graph")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--instr-steps", type=int, default=200)
    ap.add_argument("--oracle-rows", type=int, default=4)
    ap.add_argument("--steps-ref", type=int, default=None)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=("decode", "moe", "rowwise"), default="decode")
    ap.add_argument("--code", choices=("e4m3", "int8", "int8block"), default="e4m3",
                    help="rowwise workload: FP8_Dynamic (e4m3), W8A8_INT8 (int8) or block "
                         "INT8 (int8block) codes")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.steps_ref is None:
        args.steps_ref = max(1, min(args.steps, 10))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.workload == "moe":
        if world > 1 and rank != 0:
            return 0
        return run_gpu_moe(args, rank, world)
    if args.workload == "rowwise":
        if world > 1 and rank != 0:
            return 0
        return run_gpu_rowwise(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    rc = run_gpu(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
