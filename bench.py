"""Benchmark of the W8A8 block-FP8 linear hot path on GB300.

Workloads (`--workload`; the default is the largest configuration, `grid`):

  grid     the full grid: M in {1,2,4,8,16,24,32,48,64,96,128,256,512,1024,
           1536,2048,3072,4096} x (N,K) in {(1536,7168),(7168,1536),
           (4096,7168),(7168,18432),(18432,7168),(24576,7168)}, fp16 and
           bf16 out: 216 fp8bq_linear calls (activation quant + block-scaled
           GEMM, UE8M0) per pass.  Activations bf16 N(0,1) with 0.5% of the K
           channels x50, weights bf16 N(0,0.02) quantised 128x128 once,
           outside the timed region.
  decode   the decode sweep: (N,K) in {(7168,18432),(18432,7168),(4096,7168)}
           x M in {1..128} (11 points), UE8M0, bf16 out, act 1% channels x30.
  prefill  the prefill sweep: (N,K) in {(24576,7168),(4096,7168),(7168,18432)}
           x M in {256..4096} (7 points), fp32 scales, bf16 and fp32 out,
           act Student-t(3) scaled to unit RMS.
  small    M=16, N=K=1536, fp32 scales, bf16 out, fp32 N(0,0.02) weights: 100
           back-to-back calls per pass, each on its own weight copy (cold),
           and the same 100 calls on one copy (hot L2).
  quant    the standalone per-token-group quant: M in {1,64,1024,4096,16384}
           x K in {1536,7168,18432}, fp32 and UE8M0 scales; every 8th row
           holds one +-1000 spike per group.
  moe      the grouped (mixture-of-experts) linear layer (32 local experts).
  rowwise  the per-token x per-channel formats (`--code e4m3|int8|int8block`).

A step is `passes` passes over the workload's problems, replayed from one
CUDA graph; `passes` is the smallest count for which the K timed steps last
at least `--min-timed-s` seconds, so the clock samples cover a loaded GPU
whatever K is.  Every problem reads its own weight copy (and activation
copy), so the inputs of a pass are far larger than L2.

Reported beside `value`: per (M,N,K) the GEMM's time (isolated, cold; and
hot, directly after the same GEMM), TFLOPS, the pages' GB/s and the
algorithmic GB/s and the fraction of the roofline min(FP8 peak, HBM); the
two target regimes (M <= 64 against HBM, M >= 2048 against the FP8 peak);
the roofline of the dominant kernel; an end-to-end number through the same
public call with pinned host buffers; and the CPU oracle timed on a bounded
sample.  `--impl reference` times the oracle alone on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_scaled_fp8_group_gb300 import synth  # noqa: E402

METRIC = "block-FP8 GEMM µs, TFLOPS and GB/s per (M,N,K) on 1 GB300; % of roofline"
FP8_TO_BF16_NOMINAL = 2.0  # 4.5 / 2.25 PFLOP/s dense, nominal ratio
# The pages' DeepGEMM numbers on H100 80GB HBM3 ("vLLM DeepGEMM FP8 Block GEMM
# 基准测试" §3.2, DeepGEMM table), µs per (m, n, k) -- context only.
H100_DEEPGEMM_US = {
    (8, 4096, 7168): 102.9, (8, 7168, 18432): 70.8, (8, 18432, 7168): 69.3,
    (64, 4096, 7168): 69.1, (64, 7168, 18432): 69.4, (64, 18432, 7168): 70.4,
    (64, 24576, 1536): 70.1, (64, 32768, 512): 68.4, (64, 7168, 16384): 69.5,
    (128, 4096, 7168): 141.1, (128, 7168, 18432): 71.9, (128, 18432, 7168): 69.3,
    (1024, 4096, 7168): 89.7, (1024, 18432, 7168): 279.0, (2048, 4096, 7168): 175.1,
    (4096, 4096, 7168): 335.4}

OUT_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4}


# ------------------------------------------------------------- formulas

def gemm_flops(M, N, K):
    """The pages' TFLOPS numerator: 2*m*n*k ("vLLM DeepGEMM FP8 Block GEMM 基准测试"
    §4.3)."""
    return 2.0 * M * N * K


def pages_gbs_bytes(M, N, K):
    """The pages' GB/s numerator: m*k + k*n + 2*m*n ("vLLM DeepGEMM FP8 Block GEMM
    基准测试" §4.3)."""
    return M * K + K * N + 2 * M * N


def act_scale_bytes(M, K, fmt):
    """Activation scale buffer: [G][Mp] fp32, or [ceil(G/4)][Mp] packed UE8M0."""
    G, Mp = K // 128, (M + 3) // 4 * 4
    return 4 * Mp * ((G + 3) // 4 if fmt == "ue8m0" else G)


def weight_scale_bytes(N, K):
    return 4 * ((N + 127) // 128) * (K // 128)


def gemm_bytes(M, N, K, fmt="ue8m0", odt="bf16"):
    """Algorithmic bytes of one GEMM launch: e4m3 A and W, activation and
    weight scales, the output."""
    return M * K + N * K + act_scale_bytes(M, K, fmt) + weight_scale_bytes(N, K) + \
        OUT_SIZE[odt] * M * N


def linear_bytes(M, N, K, odt="bf16"):
    """Algorithmic bytes of one linear layer (quant + GEMM): bf16 A in, W,
    weight scales, the output (the intermediate codes are not counted)."""
    return 2 * M * K + N * K + weight_scale_bytes(N, K) + OUT_SIZE[odt] * M * N


def quant_bytes(M, K, fmt):
    """Activation quant: bf16 in, e4m3 codes and the scales out."""
    return 2 * M * K + M * K + act_scale_bytes(M, K, fmt)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        burst = float(d["bf16_tflops"])
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": burst,
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", burst)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def roof_time(byt, flops, peaks):
    """The roofline time max(bytes / HBM, flops / FP8 peak) and its bound."""
    fp8 = peaks["bf16_tflops"] * FP8_TO_BF16_NOMINAL
    th, tt = byt / (peaks["hbm_gbs"] * 1e9), flops / (fp8 * 1e12)
    return (th, "hbm") if th >= tt else (tt, "tensor")


def variant_name(v: dict) -> str:
    """kind/block_n/s<split>, with /mx when the tensor core applies the scales."""
    return "{kind}/{block_n}/s{split}".format(**v) + ("/mx" if v.get("mma_scale") else "")


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "block_scaled_fp8_group_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def gemm_source_hash():
    return source_hash(("gemm_impl.cuh", "gemm.cu", "ptx.cuh", "internal.h"))


def quant_source_hash():
    return source_hash(("quant.cu", "quant_math.cuh", "internal.h"))


def profile_traffic(name, src_hash):
    """DRAM traffic per algorithmic byte of the dominant kernel, from a
    committed ncu summary `profiles/<name>` taken on the current kernel
    source (sha256 prefix); None otherwise."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    t = re.search(r"traffic_per_algorithmic_byte:\s*([0-9.eE+]+)", txt)
    if not m or not t or m.group(1) != src_hash:
        return None
    return float(t.group(1))


# ------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (100 ms) from start() to stop(); start it before
    the warm-up so the samples that count are taken under load."""
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

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
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
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm_max = max(r[1] for r in rows)
        p_max = max(r[2] for r in rows)
        # under load: drawing well above idle power (the SM clock stays at its
        # maximum at idle on these parts, so it cannot tell load apart)
        loaded = [r for r in rows if r[2] > 0.4 * p_max] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in loaded])), "sm_max_mhz": sm_max,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": p_max}


# ------------------------------------------------------------- replicas

def max_over_ranks(seconds: float, device) -> float:
    """The slowest rank's time: replicas report the whole job's throughput as
    the units all ranks processed over the time of the slowest one."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def max_int_over_ranks(v: int, device) -> int:
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return int(t.item())


def job_value(units_per_rank: float, world: int, seconds: float, scale: float = 1e9) -> float:
    """Whole-job throughput of `world` replicas that each processed
    units_per_rank in `seconds` (the max over ranks): weak scaling."""
    return world * units_per_rank / seconds / scale


# ------------------------------------------------------------- workloads

class Problem:
    """One call of a linear sweep: (M, N, K), the output dtype and, for
    repeated shapes, the copy index (its own weight and activation copy)."""

    def __init__(self, M, N, K, odt, copy=0):
        self.M, self.N, self.K, self.odt, self.copy = M, N, K, odt, copy

    @property
    def key(self):  # the tensors a problem reads (shared by its output dtypes)
        return (self.M, self.N, self.K, self.copy)

    @property
    def shape(self):
        return (self.M, self.N, self.K, self.odt)


class Sweep:
    """A linear-layer workload: problems, scale format, input recipes."""

    def __init__(self, name, text, problems, fmt, act, weight, unit, act_oracle):
        self.name, self.text, self.problems, self.fmt = name, text, problems, fmt
        self.act, self.weight, self.unit, self.act_oracle = act, weight, unit, act_oracle

    def config(self, world):
        odts = sorted({p.odt for p in self.problems})
        return {"workload": self.text, "problems_per_pass": len(self.problems),
                "scale_fmt": self.fmt, "out_dtypes": odts,
                "api": "fp8bq_linear (activation quant + GEMM, two launches with PDL)",
                "l2": "inputs larger than L2: every problem reads its own weight and "
                      "activation copy",
                "parallelism": "replicas" if world > 1 else "single GPU"}

    def units(self, p):
        """Units of `value` one problem contributes."""
        if self.unit == "TFLOPS":
            return gemm_flops(p.M, p.N, p.K)
        return linear_bytes(p.M, p.N, p.K, p.odt)

    @property
    def unit_scale(self):
        return 1e12 if self.unit == "TFLOPS" else 1e9


def _weight_bf16(N, K):
    return synth.weight_bf16_blocked(N, K), "bf16"


def _weight_f32(N, K):
    return synth.normal_blocked((N, K), synth.SEED_WEIGHT, std=0.02), "fp32"


def _act_small(M, K):
    return synth.f32_to_bf16_bits_par(synth.normal_blocked((M, K), synth.SEED_ACT))


def make_sweep(name):
    if name == "grid":
        probs = [Problem(M, N, K, odt) for odt in ("bf16", "fp16") for M in synth.M_GRID
                 for (N, K) in synth.FULL_NK]
        text = ("full grid: M in {1,2,4,8,16,24,32,48,64,96,128,256,512,1024,1536,2048,3072,"
                "4096} x (N,K) in {(1536,7168),(7168,1536),(4096,7168),(7168,18432),"
                "(18432,7168),(24576,7168)}, fp16 and bf16 out; fused quant+GEMM per call; "
                "act bf16 N(0,1) 0.5% channels x50; weights bf16 N(0,0.02) 128x128; UE8M0")
        return Sweep(name, text, probs, "ue8m0", synth.act_full_grid_blocked, _weight_bf16,
                     "TFLOPS", synth.act_full_grid_blocked)
    if name == "decode":
        probs = [Problem(M, N, K, "bf16") for M in synth.DECODE_M for (N, K) in synth.DECODE_NK]
        text = ("decode sweep: (N,K) in {(7168,18432),(18432,7168),(4096,7168)} x "
                "M in {1,2,4,8,16,24,32,48,64,96,128}; act bf16 N(0,1), 1% channels x30 -> "
                "per-token-group quant (UE8M0 packed); weights bf16 N(0,0.02) 128x128 UE8M0; "
                "bf16 out")
        return Sweep(name, text, probs, "ue8m0", synth.act_decode_blocked, _weight_bf16,
                     "GB/s", synth.act_decode_blocked)
    if name == "prefill":
        probs = [Problem(M, N, K, odt) for odt in ("bf16", "fp32") for M in synth.PREFILL_M
                 for (N, K) in synth.PREFILL_NK]
        text = ("prefill sweep: (N,K) in {(24576,7168),(4096,7168),(7168,18432)} x "
                "M in {256,512,1024,1536,2048,3072,4096}; act bf16 Student-t(3) unit RMS; "
                "weights bf16 N(0,0.02) 128x128; fp32 scales; bf16 and fp32 out")
        return Sweep(name, text, probs, "fp32", synth.act_prefill_blocked, _weight_bf16,
                     "TFLOPS", synth.act_prefill_blocked)
    if name == "small":
        probs = [Problem(16, 1536, 1536, "bf16", c) for c in range(100)]
        text = ("small: M=16, N=K=1536; act bf16 N(0,1); weights fp32 N(0,0.02) 128x128; "
                "fp32 scales; bf16 out; 100 back-to-back calls per pass, each on its own "
                "weight copy")
        return Sweep(name, text, probs, "fp32", _act_small, _weight_f32, "GB/s", _act_small)
    raise ValueError(name)


# ------------------------------------------------------------- oracle legs

def oracle_weights(sweep, host_w):
    """The oracle's own quantisation of each (N,K) weight, in parallel
    threads (the C calls release the GIL); outside every timing."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    ue = sweep.fmt == "ue8m0"
    nks = sorted(host_w)

    def one(nk):
        w, kind = host_w[nk]
        return nk, oracle.quant_weight(w, oracle.BF16 if kind == "bf16" else oracle.FP32, 128,
                                       128, ue)

    with ThreadPoolExecutor(max_workers=len(nks)) as ex:
        return dict(ex.map(one, nks))


def oracle_sample(sweep, qws, rows=1):
    """Times the oracle on one thread: per (N,K), `rows` activation rows
    through oracle quant + fp64 GEMM (all N columns).  Returns (whole-pass
    seconds extrapolated linearly in M over the pass's problems, sample
    seconds, description)."""
    import oracle
    ue = sweep.fmt == "ue8m0"
    per_row, sample_s = {}, 0.0
    for (N, K) in sorted(qws):
        qw, sw = qws[(N, K)]
        xb = np.ascontiguousarray(sweep.act_oracle(rows, K))
        t0 = time.perf_counter()
        qa, sa = oracle.quant_act(xb, oracle.BF16, 128, ue)
        oracle.gemm(qa, sa, qw, sw, ue)
        dt = time.perf_counter() - t0
        sample_s += dt
        per_row[(N, K)] = dt / rows
    est = sum(per_row[(p.N, p.K)] * p.M for p in sweep.problems)
    desc = (f"{rows} activation row(s) per (N,K) through oracle quant + fp64 GEMM (all N "
            f"columns), single thread; the pass's time extrapolated linearly in M over its "
            f"{len(sweep.problems)} problems")
    return est, sample_s, desc


def oracle_all_cores(sweep, qws, threads=None):
    """The same routine over row partitions on all host cores (one row per
    thread per (N,K)); returns (extrapolated pass seconds, threads, desc)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    ue = sweep.fmt == "ue8m0"
    n = threads or os.cpu_count() or 1
    per_row = {}
    for (N, K) in sorted(qws):
        qw, sw = qws[(N, K)]
        xb = np.ascontiguousarray(sweep.act_oracle(n, K))

        def one(r):
            qa, sa = oracle.quant_act(np.ascontiguousarray(xb[r:r + 1]), oracle.BF16, 128, ue)
            oracle.gemm(qa, sa, qw, sw, ue)

        with ThreadPoolExecutor(max_workers=n) as ex:
            t0 = time.perf_counter()
            list(ex.map(one, range(n)))
            per_row[(N, K)] = (time.perf_counter() - t0) / n
    est = sum(per_row[(p.N, p.K)] * p.M for p in sweep.problems)
    return est, n, (f"{n} activation rows per (N,K), one per thread on {n} threads (row "
                    "partitions of the same single-thread oracle routine); extrapolated "
                    "linearly in M")


QUANT_TEXT = ("standalone per-token-group quant: bf16 M x K, M in {1,64,1024,4096,16384} x "
              "K in {1536,7168,18432}, group 128, N(0,1) with one +-1000 spike per group in "
              "every 8th row; fp32 scales and UE8M0 scales packed 4 per int32 (column-major, "
              "rows padded to a multiple of 4)")


def quant_problems():
    return [(M, K, fmt) for fmt in ("fp32", "ue8m0") for M in synth.QUANT_M
            for K in synth.QUANT_K]


def quant_config(world):
    return {"workload": QUANT_TEXT, "problems_per_pass": len(quant_problems()),
            "api": "fp8bq_quant_act",
            "l2": "inputs larger than L2: every (M,K) reads its own input copy",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def quant_oracle_sample(rows=64):
    import oracle
    per_row, sample_s = {}, 0.0
    for K in synth.QUANT_K:
        xb = np.ascontiguousarray(synth.act_quant_blocked(rows, K))
        for fmt in ("fp32", "ue8m0"):
            t0 = time.perf_counter()
            oracle.quant_act(xb, oracle.BF16, 128, fmt == "ue8m0")
            dt = time.perf_counter() - t0
            sample_s += dt
            per_row[(K, fmt)] = dt / rows
    est = sum(per_row[(K, fmt)] * M for (M, K, fmt) in quant_problems())
    return est, sample_s, (f"{rows} rows per (K, scale format) through the oracle quant, single "
                           "thread; extrapolated linearly in M")


# ------------------------------------------------------------- GPU helpers

def _events(torch, n, external):
    mk = (lambda: torch.cuda.Event(enable_timing=True, external=True)) if external else \
        (lambda: torch.cuda.Event(enable_timing=True))
    return [(mk(), mk()) for _ in range(n)]


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.synchronize()
    return g


def timed_steps(torch, graph, args, world, dev, local, rank):
    """W warm-up steps and K timed steps of `passes` replays each, CUDA events
    on the launching stream around every step, clocks sampled from before the
    warm-up to the end of the timed region.  Returns (mean step seconds --
    the max over ranks --, passes, clocks, wall seconds of the timed region)."""
    import torch.distributed as dist
    cal = []
    for _ in range(3):  # calibration (untimed): one pass at a time
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        cal.append(a.elapsed_time(b) / 1e3)
    pass_s = min(cal)
    passes = max(1, math.ceil(args.min_timed_s / (max(1, args.steps) * pass_s)))
    if world > 1:
        passes = max_int_over_ranks(passes, dev)
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    for _ in range(args.warmup):
        for _ in range(passes):
            graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = _events(torch, args.steps, False)
    t0 = time.perf_counter()
    for a, b in evs:
        a.record()
        for _ in range(passes):
            graph.replay()
        b.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t0
    clk = clocks.stop() if rank == 0 else None
    step_s = float(np.mean([a.elapsed_time(b) for a, b in evs])) / 1e3
    if world > 1:
        step_s = max_over_ranks(step_s, dev)
    return step_s, passes, clk, wall


def _ext_events_ok(torch):
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


class Background:
    """Runs fn() in a thread (the oracle legs, whose C calls release the GIL)
    while the GPU is kept busy."""

    def __init__(self, fn):
        self.out, self.err = None, None

        def run():
            try:
                self.out = fn()
            except BaseException as e:  # reported by result()
                self.err = e

        self.t = threading.Thread(target=run, daemon=True)
        self.t.start()

    def done(self):
        return not self.t.is_alive()

    def result(self):
        self.t.join()
        if self.err is not None:
            raise self.err
        return self.out


# ------------------------------------------------------------- linear sweeps

def run_sweep(args, rank, world, sweep):
    import torch

    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ext = _ext_events_ok(torch)
    if not ext:
        raise RuntimeError("timing needs torch.cuda.Event(external=True) (events in a graph)")
    fmt, probs = sweep.fmt, sweep.problems
    keys = sorted({p.key for p in probs})
    nks = sorted({(p.N, p.K) for p in probs})
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline

    # ---- setup (untimed): weights quantised once, one copy per problem key
    host_w, w_q, w_s = {}, {}, {}
    for (N, K) in nks:
        wh, kind = sweep.weight(N, K)
        if want_cpu:
            host_w[(N, K)] = (wh, kind)
        if kind == "bf16":
            wd = torch.from_numpy(wh.view(np.int16)).view(torch.bfloat16).to(dev)
        else:
            wd = torch.from_numpy(wh).to(dev)
        q, s = fp8bq.fp8bq_quant_weight(wd, fmt)
        del wd
        w_s[(N, K)] = s
        first = True
        for k in keys:
            if (k[1], k[2]) == (N, K):
                w_q[k] = q if first else q.clone()
                first = False
    prep = Background(lambda: oracle_weights(sweep, host_w)) if want_cpu else None
    max_m = {}
    for p in probs:
        max_m[p.K] = max(max_m.get(p.K, 0), p.M)
    host_x = {K: sweep.act(Mx, K) for K, Mx in max_m.items()}
    xs = {}
    for k in keys:
        M, N, K, _ = k
        xs[k] = torch.from_numpy(host_x[K][:M].view(np.int16)).view(torch.bfloat16).to(dev)
    outs = {p.shape + (p.copy,): torch.empty((p.M, p.N), dtype=fp8bq._CODE_TO_TORCH[
        fp8bq._dtype_code(p.odt)], device=dev) for p in probs}
    aqs, ass = {}, {}
    for k in keys:
        M, N, K, _ = k
        shape, dt = fp8bq.act_scale_shape(M, K, 128, fmt)
        aqs[k] = torch.empty((M, K), dtype=torch.uint8, device=dev)
        ass[k] = torch.empty(shape, dtype=dt, device=dev)
    ws_bytes = max(fp8bq.fp8bq_linear_workspace_bytes(p.M, p.N, p.K, fmt, p.odt) for p in probs)
    ws = torch.zeros(ws_bytes + (1 << 20), dtype=torch.uint8, device=dev)
    variants = {p.shape: fp8bq.fp8bq_select_variant(p.M, p.N, p.K, fmt, p.odt) for p in probs}
    torch.cuda.synchronize()

    def out_of(p):
        return outs[p.shape + (p.copy,)]

    def step():
        for p in probs:
            fp8bq.fp8bq_linear(xs[p.key], w_q[p.key], w_s[(p.N, p.K)], fmt=fmt,
                               out_dtype=out_of(p).dtype, out=out_of(p), workspace=ws)

    ev_i = _events(torch, len(probs), True)
    ev_b = _events(torch, len(probs), True)
    ev_h = _events(torch, len(probs), True)
    # every weight copy of each (N, K): back-to-back calls rotate over them
    copies = {}
    for k in keys:
        copies.setdefault((k[1], k[2]), []).append(w_q[k])
    R = args.b2b

    def gemm_w(p, w):
        fp8bq.fp8bq_gemm(aqs[p.key], ass[p.key], w, w_s[(p.N, p.K)], fmt=fmt,
                         out_dtype=out_of(p).dtype, out=out_of(p), workspace=ws)

    def step_b2b():
        # the pages' per-shape method: R calls of the GEMM back to back (each
        # launch overlaps the previous one's tail), events around the R calls;
        # cold: the calls rotate over the problem's weight copies
        for i, p in enumerate(probs):
            cs = copies[(p.N, p.K)]
            j0 = next(j for j, c in enumerate(cs) if c is w_q[p.key])
            ev_b[i][0].record()
            for j in range(R):
                gemm_w(p, cs[(j0 + j) % len(cs)])
            ev_b[i][1].record()

    def step_hot():
        # the same with one weight copy: operands in L2 as far as they fit
        for i, p in enumerate(probs):
            ev_h[i][0].record()
            for j in range(R):
                gemm_w(p, w_q[p.key])
            ev_h[i][1].record()

    def step_instr():
        # quant and GEMM as separate calls, events around every GEMM launch
        for i, p in enumerate(probs):
            fp8bq.fp8bq_quant_act(xs[p.key], fmt, q=aqs[p.key], s=ass[p.key])
            ev_i[i][0].record()
            fp8bq.fp8bq_gemm(aqs[p.key], ass[p.key], w_q[p.key], w_s[(p.N, p.K)], fmt=fmt,
                             out_dtype=out_of(p).dtype, out=out_of(p), workspace=ws)
            ev_i[i][1].record()

    chain_sets = {"all": list(range(len(probs)))}
    low = [i for i, p in enumerate(probs) if p.M <= 64]
    if low and len(low) < len(probs):
        chain_sets["m_le_64"] = low

    def chain_fn(idx):
        def f():
            for i in idx:
                p = probs[i]
                fp8bq.fp8bq_gemm(aqs[p.key], ass[p.key], w_q[p.key], w_s[(p.N, p.K)], fmt=fmt,
                                 out_dtype=out_of(p).dtype, out=out_of(p), workspace=ws)
        return f

    # first launches: load the table, set kernel attributes
    step()
    step_instr()
    torch.cuda.synchronize()
    g_step = capture(torch, step)
    g_instr = capture(torch, step_instr)
    g_hot = capture(torch, step_hot)
    g_b2b = capture(torch, step_b2b)
    g_chain = {name: capture(torch, chain_fn(idx)) for name, idx in chain_sets.items()}

    step_s, passes, clk, wall = timed_steps(torch, g_step, args, world, dev, local, rank)
    launches = args.steps * passes * 2 * len(probs)

    # ---- per-GEMM durations (instrumented pass), the oracle timed meanwhile
    qws = prep.result() if prep is not None else None
    cpu_job = None
    if want_cpu:
        def cpu_legs():
            est, sample_s, desc = oracle_sample(sweep, qws, rows=args.oracle_rows)
            est_all, nthr, desc_all = oracle_all_cores(sweep, qws)
            return est, sample_s, desc, est_all, nthr, desc_all
        cpu_job = Background(cpu_legs)
    gemm_ms = np.zeros(len(probs))
    n_instr = 0
    while n_instr < args.instr_passes or (cpu_job is not None and not cpu_job.done()):
        g_instr.replay()
        torch.cuda.synchronize()
        gemm_ms += np.array([a.elapsed_time(b) for a, b in ev_i])
        n_instr += 1
    event_us = gemm_ms / n_instr * 1e3
    hot_ms, b2b_ms = np.zeros(len(probs)), np.zeros(len(probs))
    for _ in range(args.instr_passes):
        g_b2b.replay()
        torch.cuda.synchronize()
        b2b_ms += np.array([a.elapsed_time(b) for a, b in ev_b])
        g_hot.replay()
        torch.cuda.synchronize()
        hot_ms += np.array([a.elapsed_time(b) for a, b in ev_h])
    gemm_us = b2b_ms / (args.instr_passes * R) * 1e3  # per call, back to back, cold
    hot_us = hot_ms / (args.instr_passes * R) * 1e3
    chain_s = {}
    for name, g in g_chain.items():
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.instr_passes):
            g.replay()
        b.record()
        b.synchronize()
        chain_s[name] = a.elapsed_time(b) / 1e3 / args.instr_passes
    assert fp8bq.fp8bq_device_status() == 0

    # ---- end to end through fp8bq_linear with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = sweep_e2e(torch, fp8bq, args, world, dev, sweep, host_x, w_q, w_s, ws, out_of)

    if rank != 0:
        return 0
    peaks = load_peaks()
    fp8 = peaks["bf16_tflops"] * FP8_TO_BF16_NOMINAL
    fp8_sus = peaks["bf16_tflops_sustained"] * FP8_TO_BF16_NOMINAL
    per = []
    for i, p in enumerate(probs):
        t = gemm_us[i] * 1e-6
        byt = gemm_bytes(p.M, p.N, p.K, fmt, p.odt)
        fl = gemm_flops(p.M, p.N, p.K)
        tr, bound = roof_time(byt, fl, peaks)
        per.append({"m": p.M, "n": p.N, "k": p.K, "out": p.odt, "copy": p.copy,
                    "us": gemm_us[i], "us_hot": hot_us[i], "us_event": event_us[i],
                    "tflops": fl / t / 1e12,
                    "gbs_pages": pages_gbs_bytes(p.M, p.N, p.K) / t / 1e9,
                    "gbs_alg": byt / t / 1e9, "roofline_frac": tr / t, "bound": bound,
                    "variant": variant_name(variants[p.shape]),
                    "h100_deepgemm_us": H100_DEEPGEMM_US.get((p.M, p.N, p.K))})
    per = merge_copies(per)

    def regime(sel, kind):
        rows = [(i, p) for i, p in enumerate(probs) if sel(p)]
        if not rows:
            return None
        t = sum(gemm_us[i] for i, _ in rows) * 1e-6
        if kind == "hbm":
            byt = sum(gemm_bytes(p.M, p.N, p.K, fmt, p.odt) for _, p in rows)
            fr = [gemm_bytes(p.M, p.N, p.K, fmt, p.odt) / (peaks["hbm_gbs"] * 1e9) /
                  (gemm_us[i] * 1e-6) for i, p in rows]
            out = {"gemms": len(rows), "gbs_alg": byt / t / 1e9, "peak_gbs": peaks["hbm_gbs"],
                   "frac": byt / t / 1e9 / peaks["hbm_gbs"], "frac_min": min(fr),
                   "frac_max": max(fr), "peak_source": "measured copy bandwidth"}
            if "m_le_64" in chain_s and sel is _m_le_64:
                out["frac_chained"] = byt / chain_s["m_le_64"] / 1e9 / peaks["hbm_gbs"]
                out["chain_us"] = chain_s["m_le_64"] * 1e6
            return out
        fl = sum(gemm_flops(p.M, p.N, p.K) for _, p in rows)
        fr = [gemm_flops(p.M, p.N, p.K) / (fp8 * 1e12) / (gemm_us[i] * 1e-6) for i, p in rows]
        return {"gemms": len(rows), "tflops": fl / t / 1e12, "peak_tflops": fp8,
                "frac": fl / t / 1e12 / fp8, "frac_min": min(fr), "frac_max": max(fr),
                "frac_of_sustained": fl / t / 1e12 / fp8_sus,
                "peak_source": "2 x measured bf16 cuBLAS burst (nominal fp8/bf16 ratio); "
                               "frac_of_sustained against 2 x the sustained bf16 figure"}

    targets = {"m_le_64_vs_hbm": regime(_m_le_64, "hbm"),
               "m_ge_2048_vs_fp8": regime(lambda p: p.M >= 2048, "tensor")}

    # the dominant kernel class: the GEMM launches of the bound that holds
    # most of the instrumented time
    cls = {"hbm": [], "tensor": []}
    for i, p in enumerate(probs):
        byt = gemm_bytes(p.M, p.N, p.K, fmt, p.odt)
        cls[roof_time(byt, gemm_flops(p.M, p.N, p.K), peaks)[1]].append(i)
    dom = max(cls, key=lambda c: sum(gemm_us[i] for i in cls[c]))
    idx = cls[dom]
    t_dom = sum(gemm_us[i] for i in idx) * 1e-6
    names = sorted({variant_name(variants[probs[i].shape]) for i in idx})
    n_mx = sum(1 for i in idx if variants[probs[i].shape]["mma_scale"])
    kern = (f"block-scaled FP8 GEMM, {len(idx)} {dom}-bound launches of the pass "
            f"({n_mx} gemm_mx_kernel, {len(idx) - n_mx} gemm_kernel; variants "
            f"{', '.join(names[:12])}{' ...' if len(names) > 12 else ''})")
    alg_bytes_dom = sum(gemm_bytes(probs[i].M, probs[i].N, probs[i].K, fmt, probs[i].odt)
                        for i in idx)
    ratio = profile_traffic(f"gemm_{sweep.name}_traffic.txt", gemm_source_hash())
    traffic = None if ratio is None else ratio * alg_bytes_dom / len(idx)
    if dom == "tensor":
        fl = sum(gemm_flops(probs[i].M, probs[i].N, probs[i].K) for i in idx)
        ach = fl / t_dom / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": fp8_sus, "unit": "TFLOP/s",
                "frac": ach / fp8_sus, "traffic": traffic,
                "frac_of_burst_peak": ach / fp8,
                "peak_source": f"{peaks['source']}: 2 x bf16_tflops_sustained (the kernel is "
                               "timed inside a seconds-long loop; nominal fp8/bf16 ratio 2)"}
    else:
        ach = alg_bytes_dom / t_dom / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy)"}
        if len(chain_sets["all"]) == len(idx):
            roof["achieved_chained"] = alg_bytes_dom / chain_s["all"] / 1e9
            roof["frac_chained"] = roof["achieved_chained"] / peaks["hbm_gbs"]
    roof.update({"kernel": kern, "launches_per_pass": len(idx),
                 "algorithmic_bytes_per_launch": alg_bytes_dom / len(idx),
                 "method": "achieved = the class's algorithmic flops (or bytes) over the sum "
                           "of its launches' durations, each GEMM timed per call over "
                           f"{R} back-to-back calls in a graph that rotate over the "
                           "problem's weight copies (cold), CUDA events on the launching "
                           "stream; traffic = the ncu DRAM bytes per algorithmic byte of the "
                           "committed summary x the class's bytes per launch"})

    cpu = None
    if cpu_job is not None:
        est, sample_s, desc, est_all, nthr, desc_all = cpu_job.result()
        units = sum(sweep.units(p) for p in probs)
        cpu = {"value": units / est / sweep.unit_scale, "unit": sweep.unit, "cores": 1,
               "kind": "oracle", "extrapolated": True,
               "sample": desc + f" (sample took {sample_s:.1f} s; run while the GPU's "
                                "per-GEMM passes ran)",
               "all_cores": {"value": units / est_all / sweep.unit_scale, "unit": sweep.unit,
                             "cores": nthr, "sample": desc_all}}
    units_pass = sum(sweep.units(p) for p in probs)
    value = job_value(units_pass * passes, world, step_s, sweep.unit_scale)
    t_roof_pass = sum(roof_time(linear_bytes(p.M, p.N, p.K, p.odt), gemm_flops(p.M, p.N, p.K),
                                peaks)[0] for p in probs)
    line = {
        "metric": METRIC, "value": value, "unit": sweep.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic", "config": sweep.config(world),
        "passes_per_step": passes,
        "timing": "graph replays; a step = passes_per_step passes over the problems (the "
                  "smallest count that makes the timed region >= --min-timed-s); CUDA events "
                  "on the launching stream around every step; 3 untimed calibration passes "
                  "before the warm-up.  per_shape: us = per call over back-to-back calls of "
                  "the GEMM rotating over the problem's weight copies (the pages' per-shape "
                  "method: warm-up, then the mean of many calls), us_hot = the same on one "
                  "weight copy, us_event = the GEMM alone between CUDA events after its quant "
                  "(includes the launch gap a graph node pays)",
        "step_roofline_frac": t_roof_pass * passes / step_s,
        "roofline": roof, "targets": targets, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches, "clocks": clk,
        "gemm_chain_us": {k: v * 1e6 for k, v in chain_s.items()},
        "instrumented_passes": n_instr, "per_shape": per, "wall_timed_s": wall,
        "gemm_source_sha256_16": gemm_source_hash(),
    }
    print(json.dumps(_round(line)), flush=True)
    return 0


def _m_le_64(p):
    return p.M <= 64


def merge_copies(per):
    """One entry per (m, n, k, out): the mean over the problem's copies."""
    groups = {}
    for e in per:
        groups.setdefault((e["m"], e["n"], e["k"], e["out"]), []).append(e)
    out = []
    for key, es in groups.items():
        e = dict(es[0])
        e.pop("copy")
        for f in ("us", "us_hot", "us_event", "tflops", "gbs_pages", "gbs_alg", "roofline_frac"):
            e[f] = float(np.mean([x[f] for x in es]))
        if len(es) > 1:
            e["copies"] = len(es)
        out.append(e)
    return out


def _round(o):
    if isinstance(o, float):
        return float(f"{o:.6g}")
    if isinstance(o, dict):
        return {k: _round(v) for k, v in o.items()}
    if isinstance(o, list):
        return [_round(v) for v in o]
    return o


def sweep_e2e(torch, fp8bq, args, world, dev, sweep, host_x, w_q, w_s, ws, out_of):
    """fp8bq_linear per problem with every input copied in from pinned host
    memory and every output copied back, each step.  The copies overlap the
    compute: the step runs the problems largest output first, so the
    device-to-host copies (the larger direction) start early and stream while
    the rest computes; inputs go up on one side stream in the same order, and
    the compute stream waits for the next inputs once per group of up to 6
    problems and 16 MB (each cross-stream wait cuts the chain of programmatic
    launches); outputs go back on another side stream as each layer ends."""
    probs, fmt = sweep.problems, sweep.fmt
    hx = {K: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
          for K, v in host_x.items()}
    xd = {i: torch.empty((p.M, p.K), dtype=torch.bfloat16, device=dev)
          for i, p in enumerate(probs)}
    ho = {i: torch.empty(out_of(p).shape, dtype=out_of(p).dtype).pin_memory()
          for i, p in enumerate(probs)}
    h2d = sum(2 * p.M * p.K for p in probs)
    d2h = sum(OUT_SIZE[p.odt] * p.M * p.N for p in probs)
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    order = sorted(range(len(probs)),
                   key=lambda i: -OUT_SIZE[probs[i].odt] * probs[i].M * probs[i].N)
    # wait groups: up to 6 problems and 16 MB of inputs per cross-stream wait
    groups, j = [], 0
    while j < len(order):
        k, byt = j, 0
        while k < len(order) and k - j < 6:
            b = 2 * probs[order[k]].M * probs[order[k]].K
            if k > j and byt + b > (16 << 20):
                break
            byt += b
            k += 1
        groups.append((j, k))
        j = k

    def e2e_step():
        cur = torch.cuda.current_stream()
        h2d_s.wait_stream(cur)
        d2h_s.wait_stream(cur)
        ready = []
        with torch.cuda.stream(h2d_s):
            for i in order:
                p = probs[i]
                xd[i].copy_(hx[p.K][:p.M], non_blocking=True)
                e = torch.cuda.Event()
                e.record(h2d_s)
                ready.append(e)
        for (j0, j1) in groups:
            cur.wait_event(ready[j1 - 1])
            for i in order[j0:j1]:
                p = probs[i]
                o = out_of(p)
                fp8bq.fp8bq_linear(xd[i], w_q[p.key], w_s[(p.N, p.K)], fmt=fmt,
                                   out_dtype=o.dtype, out=o, workspace=ws)
                done = torch.cuda.Event()
                done.record(cur)
                d2h_s.wait_event(done)
                with torch.cuda.stream(d2h_s):
                    ho[i].copy_(o, non_blocking=True)
        cur.wait_stream(h2d_s)
        cur.wait_stream(d2h_s)

    e2e_step()
    torch.cuda.synchronize()
    g = capture(torch, e2e_step)
    for _ in range(max(1, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, args.e2e_steps))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        g.replay()
    b.record()
    b.synchronize()
    s = a.elapsed_time(b) / 1e3 / n
    if world > 1:
        s = max_over_ranks(s, dev)
    units = sum(sweep.units(p) for p in probs)
    return {"value": job_value(units, world, s, sweep.unit_scale), "unit": sweep.unit,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": s * 1e3,
            "steps": n, "passes_per_step": 1,
            "api": "fp8bq_linear per problem (graph), largest output first; every step copies "
                   "each problem's input from pinned host memory on a side stream ahead of its "
                   "layer (the compute waits once per group of up to 6 problems and 16 MB) and "
                   "its output back on another side stream"}


# ------------------------------------------------------------- quant workload

def run_quant(args, rank, world):
    import torch

    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    probs = quant_problems()
    base = {K: synth.act_quant_blocked(max(synth.QUANT_M), K) for K in synth.QUANT_K}
    xs = {(M, K): torch.from_numpy(base[K][:M].view(np.int16)).view(torch.bfloat16).to(dev)
          for (M, K, _) in probs}
    qs, ss = {}, {}
    for (M, K, fmt) in probs:
        shape, dt = fp8bq.act_scale_shape(M, K, 128, fmt)
        qs[(M, K, fmt)] = torch.empty((M, K), dtype=torch.uint8, device=dev)
        ss[(M, K, fmt)] = torch.empty(shape, dtype=dt, device=dev)

    # extra input copies for the back-to-back per-shape measurement (cold:
    # calls rotate over copies that together exceed the L2)
    xcopies = {}
    for (M, K) in xs:
        n = min(8, max(2, -(-(400 << 20) // (2 * M * K))))
        xcopies[(M, K)] = [xs[(M, K)]] + [xs[(M, K)].clone() for _ in range(n - 1)]
    R = args.b2b

    def call(p, x=None):
        M, K, fmt = p
        fp8bq.fp8bq_quant_act(xs[(M, K)] if x is None else x, fmt, q=qs[p], s=ss[p])

    def step():
        for p in probs:
            call(p)

    ev_i = _events(torch, len(probs), True)
    ev_h = _events(torch, len(probs), True)

    def step_instr():
        for i, p in enumerate(probs):
            ev_i[i][0].record()
            call(p)
            ev_i[i][1].record()

    ev_b = _events(torch, len(probs), True)

    def step_b2b():
        for i, p in enumerate(probs):
            cs = xcopies[(p[0], p[1])]
            ev_b[i][0].record()
            for j in range(R):
                call(p, cs[j % len(cs)])
            ev_b[i][1].record()

    def step_hot():
        for i, p in enumerate(probs):
            ev_h[i][0].record()
            for j in range(R):
                call(p)
            ev_h[i][1].record()

    step()
    torch.cuda.synchronize()
    g_step, g_instr = capture(torch, step), capture(torch, step_instr)
    g_hot, g_b2b = capture(torch, step_hot), capture(torch, step_b2b)
    step_s, passes, clk, wall = timed_steps(torch, g_step, args, world, dev, local, rank)
    cpu_job = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_job = Background(lambda: quant_oracle_sample(args.oracle_rows * 16))
    ev_us = np.zeros(len(probs))
    n_instr = 0
    while n_instr < args.instr_passes or (cpu_job is not None and not cpu_job.done()):
        g_instr.replay()
        torch.cuda.synchronize()
        ev_us += np.array([a.elapsed_time(b) for a, b in ev_i]) * 1e3
        n_instr += 1
    ev_us /= n_instr
    us, hot = np.zeros(len(probs)), np.zeros(len(probs))
    for _ in range(args.instr_passes):
        g_b2b.replay()
        torch.cuda.synchronize()
        us += np.array([a.elapsed_time(b) for a, b in ev_b]) * 1e3
        g_hot.replay()
        torch.cuda.synchronize()
        hot += np.array([a.elapsed_time(b) for a, b in ev_h]) * 1e3
    us /= args.instr_passes * R
    hot /= args.instr_passes * R
    assert fp8bq.fp8bq_device_status() == 0

    e2e = None
    if not args.no_e2e:
        hx = {K: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
              for K, v in base.items()}
        xd = {p: torch.empty((p[0], p[1]), dtype=torch.bfloat16, device=dev) for p in probs}
        hq = {p: torch.empty(qs[p].shape, dtype=torch.uint8).pin_memory() for p in probs}
        hs = {p: torch.empty(ss[p].shape, dtype=ss[p].dtype).pin_memory() for p in probs}
        h2d = sum(2 * M * K for (M, K, _) in probs)
        d2h = sum(M * K + act_scale_bytes(M, K, f) for (M, K, f) in probs)

        def e2e_step():
            for p in probs:
                M, K, fmt = p
                xd[p].copy_(hx[K][:M], non_blocking=True)
                fp8bq.fp8bq_quant_act(xd[p], fmt, q=qs[p], s=ss[p])
                hq[p].copy_(qs[p], non_blocking=True)
                hs[p].copy_(ss[p], non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        g = capture(torch, e2e_step)
        for _ in range(max(1, args.warmup)):
            g.replay()
        torch.cuda.synchronize()
        n = max(1, min(args.steps, args.e2e_steps))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            g.replay()
        b.record()
        b.synchronize()
        s = a.elapsed_time(b) / 1e3 / n
        if world > 1:
            s = max_over_ranks(s, dev)
        e2e = {"value": job_value(sum(quant_bytes(*p) for p in probs), world, s), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": s * 1e3,
               "steps": n, "api": "fp8bq_quant_act per problem (graph), input copied in from "
                                  "pinned host memory, codes and scales copied back, serially"}
    if rank != 0:
        return 0
    peaks = load_peaks()
    per = []
    for i, (M, K, fmt) in enumerate(probs):
        b = quant_bytes(M, K, fmt)
        per.append({"m": M, "k": K, "scale_fmt": fmt, "us": us[i], "us_hot": hot[i],
                    "us_event": ev_us[i],
                    "gbs_alg": b / (us[i] * 1e-6) / 1e9,
                    "roofline_frac": b / (peaks["hbm_gbs"] * 1e9) / (us[i] * 1e-6)})
    tot = sum(quant_bytes(*p) for p in probs)
    ach = tot / (us.sum() * 1e-6) / 1e9
    ratio = profile_traffic("quant_act_traffic.txt", quant_source_hash())
    roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"],
            "traffic": None if ratio is None else ratio * tot / len(probs),
            "kernel": f"quant_act_kernel, {len(probs)} launches per pass",
            "algorithmic_bytes_per_launch": tot / len(probs),
            "method": "achieved = the pass's algorithmic bytes over the sum of the launches' "
                      "durations, each timed per call over back-to-back calls in a graph "
                      "that rotate over input copies larger than the L2 together",
            "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy)"}
    by_fmt = {}
    for fmt in ("fp32", "ue8m0"):
        sel = [i for i, p in enumerate(probs) if p[2] == fmt and p[0] >= 4096]
        b = sum(quant_bytes(*probs[i]) for i in sel)
        by_fmt[fmt] = {"m_ge_4096_frac": b / (sum(us[i] for i in sel) * 1e-6) / 1e9 /
                       peaks["hbm_gbs"]}
    cpu = None
    if cpu_job is not None:
        est, sample_s, desc = cpu_job.result()
        cpu = {"value": tot / est / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "extrapolated": True, "sample": desc + f" (sample took {sample_s:.2f} s)"}
    line = {
        "metric": METRIC, "value": job_value(tot * passes, world, step_s), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic", "config": quant_config(world),
        "passes_per_step": passes,
        "timing": "graph replays; a step = passes_per_step passes over the 30 quant calls; "
                  "CUDA events on the launching stream around every step.  per_shape: us = "
                  "per call over back-to-back calls rotating over input copies (cold), "
                  "us_hot = on one copy, us_event = one call between CUDA events",
        "roofline": roof, "targets": by_fmt, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": args.steps * passes * len(probs), "clocks": clk, "per_shape": per,
        "wall_timed_s": wall, "quant_source_sha256_16": quant_source_hash(),
    }
    print(json.dumps(_round(line)), flush=True)
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


def run_gpu_moe(args, rank, world):
    import torch

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

    ev = _events(torch, len(probs), True)

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
    g1, g2 = capture(torch, step), capture(torch, step_split)
    step_s, passes, clk, wall = timed_steps(torch, g1, args, 1, dev, local, rank)
    gemm_ms = np.zeros(len(probs))
    for _ in range(args.instr_passes):
        g2.replay()
        torch.cuda.synchronize()
        gemm_ms += np.array([a.elapsed_time(b) for a, b in ev])
    gemm_us = gemm_ms / args.instr_passes * 1e3
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
    g3 = capture(torch, e2e_step)
    for _ in range(max(1, args.warmup)):
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
    per = []
    for i, (T, N, K, counts, M_max) in enumerate(probs):
        t = gemm_us[i] * 1e-6
        byt = moe_bytes(N, K, counts, False)
        fl = 2.0 * int(counts.sum()) * N * K
        tr, bound = roof_time(byt, fl, peaks)
        per.append({"tokens": T, "n": N, "k": K, "experts": E, "m_max": M_max,
                    "experts_with_tokens": int((counts > 0).sum()),
                    "token_rows": int(counts.sum()), "us": gemm_us[i],
                    "tflops": fl / t / 1e12, "gbs_alg": byt / t / 1e9,
                    "roofline_frac": tr / t, "bound": bound,
                    "variant": variant_name(variants[i])})
    tot_gemm = sum(moe_bytes(p[1], p[2], p[3], False) for p in probs)
    achieved = tot_gemm / (gemm_us.sum() * 1e-6) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        est, sample_s, desc = moe_oracle_sample()
        cpu = {"value": step_total / est / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "extrapolated": True, "sample": desc + f" (sample took {sample_s:.1f} s)"}
    line = {
        "metric": METRIC, "value": step_total * passes / step_s / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": MOE_WORKLOAD, "problems_per_pass": len(probs),
                   "l2": "inputs larger than L2: every problem reads its own weight copy "
                         "(0.47-0.94 GB each)",
                   "parallelism": "single GPU"},
        "passes_per_step": passes,
        "timing": "graph: a pass = fp8bq_grouped_linear per problem; a step = passes_per_step "
                  "passes; per-GEMM durations from an instrumented pass",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                     "kernel": "grouped block-FP8 GEMM (gemm_kernel / gemm_mx_kernel, grouped "
                               "tiles), 4 launches per pass",
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy)"},
        "cpu_baseline": cpu,
        "e2e": {"value": step_total / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3, "steps": n_e2e,
                "api": "fp8bq_grouped_linear per problem (graph), activations and counts "
                       "copied in from pinned host memory and outputs copied back each step"},
        "gpu_launches": args.steps * passes * 2 * len(probs), "clocks": clk, "per_shape": per,
        "wall_timed_s": wall, "gemm_source_sha256_16": gemm_source_hash(),
    }
    print(json.dumps(_round(line)), flush=True)
    return 0


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


def rowwise_problems():
    return [(M, N, K) for M in synth.DECODE_M for (N, K) in synth.DECODE_NK]


def rowwise_oracle_sample(code):
    """The oracle on one thread over one activation row per (N,K) of the
    rowwise workload, extrapolated linearly in M."""
    import oracle
    est, sample_s = 0.0, 0.0
    for (N, K) in synth.DECODE_NK:
        wb = synth.weight_bf16_blocked(N, K)
        xb = synth.act_decode(1, K)
        if code == "int8block":
            qw, sw = oracle.quant_weight_int8(wb, oracle.BF16)
            t0 = time.perf_counter()
            qa, sa = oracle.quant_act_int8(xb, oracle.BF16)
            oracle.gemm_int8_block(qa, sa, qw, sw)
        else:
            i8 = code == "int8"
            qw, sw = oracle.quant_rows(wb, oracle.BF16, int8=i8)
            t0 = time.perf_counter()
            qa, sa = oracle.quant_rows(xb, oracle.BF16, int8=i8)
            oracle.gemm_rowcol(qa, sa, qw, sw, i8)
        dt = time.perf_counter() - t0
        sample_s += dt
        est += dt * sum(synth.DECODE_M)
    return est, sample_s, ("one activation row per (N,K) through the oracle's quant and GEMM, "
                           "single thread; extrapolated linearly in M")


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
    probs = rowwise_problems()
    w_q, w_s = {}, {}
    for (N, K) in synth.DECODE_NK:
        wd = torch.from_numpy(synth.weight_bf16_blocked(N, K).view(np.int16)).view(
            torch.bfloat16).to(dev)
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
    ev = _events(torch, len(probs), True)

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
    g1, g2 = capture(torch, step), capture(torch, step_split)
    step_s, passes, clk, wall = timed_steps(torch, g1, args, 1, dev, local, rank)
    gemm_ms = np.zeros(len(probs))
    for _ in range(args.instr_passes):
        g2.replay()
        torch.cuda.synchronize()
        gemm_ms += np.array([a.elapsed_time(b) for a, b in ev])
    gemm_us = gemm_ms / args.instr_passes * 1e3
    assert fp8bq.fp8bq_device_status() == 0

    # large M: the GEMM alone, two weight copies alternating (each > L2 / 2)
    prefill = []
    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_TO_BF16_NOMINAL
    for (N, K) in synth.DECODE_NK:
        wq2 = [w_q[(1, N, K)], w_q[(2, N, K)]]
        for M in ROWWISE_PREFILL_M:
            xa = torch.from_numpy(synth.act_prefill_blocked(M, K).view(np.int16)).view(
                torch.bfloat16).to(dev)
            aq, as_ = fc.quant_a(xa)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsz = fc.gemm_ws(M, N, K)
            wsp = ws if wsz <= ws.numel() else torch.zeros(wsz, dtype=torch.uint8, device=dev)
            for i in range(3):
                fc.gemm(aq, as_, wq2[i % 2], w_s[(N, K)], o, wsp)
            reps = 10
            evs = _events(torch, reps, False)
            for i in range(reps):
                evs[i][0].record()
                fc.gemm(aq, as_, wq2[i % 2], w_s[(N, K)], o, wsp)
                evs[i][1].record()
            torch.cuda.synchronize()
            us = float(np.median([a.elapsed_time(b) for a, b in evs])) * 1e3
            fl = gemm_flops(M, N, K)
            entry = {"m": M, "n": N, "k": K, "us": us, "tflops": fl / us / 1e6,
                     "variant": variant_name(fc.select(M, N, K))}
            if code == "e4m3":
                entry["frac_of_fp8_peak"] = fl / us / 1e6 / fp8_peak
            prefill.append(entry)
            del xa, aq, as_, o
    assert fp8bq.fp8bq_device_status() == 0

    per = []
    for i, (M, N, K) in enumerate(probs):
        t = gemm_us[i] * 1e-6
        b = fc.gemm_bytes(M, N, K)
        per.append({"m": M, "n": N, "k": K, "us": gemm_us[i],
                    "tflops": gemm_flops(M, N, K) / t / 1e12, "gbs_alg": b / t / 1e9,
                    "roofline_frac": b / (peaks["hbm_gbs"] * 1e9) / t,
                    "variant": variant_name(variants[(M, N, K)])})
    tot = sum(fc.gemm_bytes(*p) for p in probs)
    achieved = tot / (gemm_us.sum() * 1e-6) / 1e9
    step_total = sum(fc.step_bytes(*p) for p in probs)
    kern = {"e4m3": "gemm_mx_kernel (rowwise: plain kind::f8f6f4, scales in the epilogue)",
            "int8": "gemm_i8_kernel (mma.sync m16n8k32 s8, TMA-fed) or gemm_mx_kernel on two "
                    "e4m3 planes, per shape from the measured table",
            "int8block": "gemm_i8_kernel (block promotion per K slab, mma.sync m16n8k32 s8) or "
                         "gemm_mx_kernel on two e4m3 planes, per shape from the measured table"}[code]
    cpu = None
    if not args.no_cpu_baseline:
        est, sample_s, desc = rowwise_oracle_sample(code)
        cpu = {"value": step_total / est / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "extrapolated": True, "sample": desc + f" (sample took {sample_s:.1f} s)"}
    line = {
        "metric": METRIC, "value": step_total * passes / step_s / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": code, "data": "synthetic",
        "config": {"workload": ROWWISE_WORKLOAD.format(
                       code=code, aq=ROWWISE_QUANT[code][0], wq=ROWWISE_QUANT[code][1],
                       api=ROWWISE_QUANT[code][2]),
                   "problems_per_pass": len(probs),
                   "l2": "inputs larger than L2: each GEMM reads its own weight copy",
                   "parallelism": "single GPU"},
        "passes_per_step": passes,
        "timing": "graph: a pass = one linear call per problem; a step = passes_per_step "
                  "passes; per-GEMM durations from an instrumented pass",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": None, "kernel": kern,
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy)"},
        "cpu_baseline": cpu, "e2e": None,
        "gpu_launches": args.steps * passes * 2 * len(probs), "clocks": clk, "per_shape": per,
        "prefill_gemm": prefill, "wall_timed_s": wall, "gemm_source_sha256_16": gemm_source_hash(),
    }
    print(json.dumps(_round(line)), flush=True)
    return 0


# ------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The oracle (the CPU reference of this path) on the host cores, on the
    GPU arm's workload, config, metric and unit: every step times a bounded
    sample of the workload and extrapolates it to the whole step."""
    if rank != 0:
        return 0
    w = args.workload
    if w in ("grid", "decode", "prefill", "small"):
        sweep = make_sweep(w)
        host_w = {(N, K): sweep.weight(N, K) for (N, K) in sorted({(p.N, p.K)
                                                                   for p in sweep.problems})}
        qws = oracle_weights(sweep, host_w)
        one = lambda: oracle_sample(sweep, qws, rows=1)  # noqa: E731
        units = sum(sweep.units(p) for p in sweep.problems)
        unit, scale, config = sweep.unit, sweep.unit_scale, sweep.config(world)
    elif w == "quant":
        one = lambda: quant_oracle_sample(16)  # noqa: E731
        units = sum(quant_bytes(*p) for p in quant_problems())
        unit, scale, config = "GB/s", 1e9, quant_config(world)
    elif w == "moe":
        one = moe_oracle_sample
        units = sum(moe_bytes(p[1], p[2], p[3], True) for p in moe_problems())
        unit, scale = "GB/s", 1e9
        config = {"workload": MOE_WORKLOAD, "problems_per_pass": len(moe_problems()),
                  "l2": "inputs larger than L2: every problem reads its own weight copy "
                        "(0.47-0.94 GB each)", "parallelism": "single GPU"}
    else:
        one = lambda: rowwise_oracle_sample(args.code)  # noqa: E731
        probs = rowwise_problems()
        fc_bytes = block_int8_step_bytes if args.code == "int8block" else rowwise_step_bytes
        units = sum(fc_bytes(*p) for p in probs)
        unit, scale = "GB/s", 1e9
        config = {"workload": ROWWISE_WORKLOAD.format(
                      code=args.code, aq=ROWWISE_QUANT[args.code][0],
                      wq=ROWWISE_QUANT[args.code][1], api=ROWWISE_QUANT[args.code][2]),
                  "problems_per_pass": len(probs),
                  "l2": "inputs larger than L2: each GEMM reads its own weight copy",
                  "parallelism": "single GPU"}
    for _ in range(args.warmup):
        one()
    ests, samples = [], []
    desc = ""
    t0 = time.perf_counter()
    for _ in range(args.steps):
        est, sample_s, desc = one()
        ests.append(est)
        samples.append(sample_s)
    wall = time.perf_counter() - t0
    est = float(np.mean(ests))
    value = units / est / scale
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": est * 1e3,
        "extrapolated": True, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": config, "passes_per_step": 1,
        "timing": "every step times the oracle on a bounded sample of the workload (one "
                  "activation row per (N,K), single thread) and extrapolates linearly in M to "
                  "one pass; ms_per_step is that extrapolation, wall_s the time the samples "
                  "took",
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "sample_s_per_step": float(np.mean(samples)), "wall_s": wall,
    }
    print(json.dumps(_round(line)), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("fp8bq", "reference"), default="fp8bq")
    ap.add_argument("--workload", choices=("grid", "decode", "prefill", "small", "quant", "moe",
                                           "rowwise"), default="grid")
    ap.add_argument("--code", choices=("e4m3", "int8", "int8block"), default="e4m3",
                    help="rowwise workload: FP8_Dynamic (e4m3), W8A8_INT8 (int8) or block "
                         "INT8 (int8block) codes")
    ap.add_argument("--min-timed-s", type=float, default=20.0,
                    help="passes per step are chosen so the K timed steps last at least this")
    ap.add_argument("--instr-passes", type=int, default=10)
    ap.add_argument("--b2b", type=int, default=8,
                    help="back-to-back calls per problem in the per-shape measurement")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--oracle-rows", type=int, default=24)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.workload in ("moe", "rowwise"):
        if world > 1 and rank != 0:
            return 0
        return (run_gpu_moe if args.workload == "moe" else run_gpu_rowwise)(args, rank, 1)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    if args.workload == "quant":
        rc = run_quant(args, rank, world)
    else:
        rc = run_sweep(args, rank, world, make_sweep(args.workload))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
