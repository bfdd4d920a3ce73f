"""Seeded synthetic inputs for the W8A8 block-FP8 linear path.

This module only draws random numbers and shapes them into the workloads'
value distributions; it holds none of the quantisation or GEMM arithmetic.
It is the one module that both the CUDA path's tests/benchmark and the CPU
oracle's tests read their inputs from.

All draws use numpy's PCG64 generator (``numpy.random.default_rng(seed)``),
which gives the same stream on x86_64 and aarch64.  Activations are returned
as bf16/fp16 bit patterns (uint16) rounded to nearest-even from fp32;
weights as fp32 or bf16 bits.

Workload recipes (the shapes the pages benchmark; DeepSeek-V3 projection
N/K, "vLLM 量化 Kernel 配置机制" §3.2 and "vLLM DeepGEMM FP8 Block GEMM 基准测试"
§3.2):
  small      M=16, N=K=1536: act N(0,1) seed 0; weight fp32 N(0,0.02) seed 1
  decode     act N(0,1), 1% of K-channels x30; weight N(0,0.02)
  prefill    act Student-t(nu=3) scaled to unit RMS; weight N(0,0.02)
  quant      act N(0,1); every 8th row (m % 8 == 3) holds one +-1000 spike per
             128-group (position and sign seeded)
  full grid  act N(0,1), 0.5% of K-channels x50; weight N(0,0.02)
  moe        grouped GEMM: tokens routed top-k over E_total experts with a
             seeded popularity (Dirichlet(0.5) over the experts), counts of
             the first E local experts; per expert act as decode (1% of
             K-channels x30), weights N(0,0.02) seeded per expert
"""
from __future__ import annotations

import numpy as np

SEED_ACT = 0
SEED_WEIGHT = 1
SEED_STRUCT = 2  # outlier channels / spike positions


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 bit patterns (numpy's cast rounds to nearest even)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _row_blocks(shape, block_rows):
    rows = shape[0]
    return [(b, slice(r, min(rows, r + block_rows)))
            for b, r in enumerate(range(0, rows, block_rows))]


def _par_map(fn, items, threads=None):
    from concurrent.futures import ThreadPoolExecutor
    import os
    with ThreadPoolExecutor(max_workers=threads or min(16, os.cpu_count() or 1)) as ex:
        return list(ex.map(fn, items))


def normal_blocked(shape, seed: int, std: float = 1.0, block_rows: int = 1024) -> np.ndarray:
    """N(0, std^2) fp32 drawn in blocks of `block_rows` rows, block b from its
    own PCG64 stream seeded with SeedSequence([seed, b]), filled by parallel
    threads.  A different (but equally seeded and reproducible) recipe from
    `normal`, for the benchmark's multi-GB inputs; the values of a row depend
    only on (seed, row), not on the number of rows drawn."""
    x = np.empty(shape, dtype=np.float32)

    def fill(item):
        b, rows = item
        np.random.default_rng([seed, b]).standard_normal(size=x[rows].shape, dtype=np.float32,
                                                         out=x[rows])
        if std != 1.0:
            x[rows] *= np.float32(std)

    _par_map(fill, _row_blocks(shape, block_rows))
    return x


def f32_to_bf16_bits_par(x: np.ndarray, block_rows: int = 1024) -> np.ndarray:
    """`f32_to_bf16_bits` over row blocks in parallel threads (same bits)."""
    out = np.empty(x.shape, dtype=np.uint16)

    def conv(item):
        _, rows = item
        out[rows] = f32_to_bf16_bits(x[rows])

    _par_map(conv, _row_blocks(x.shape, block_rows))
    return out


def normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    x = _rng(seed).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def student_t_unit_rms(shape, seed: int, nu: float = 3.0) -> np.ndarray:
    t = _rng(seed).standard_t(nu, size=shape)
    rms = np.sqrt(np.mean(np.square(t, dtype=np.float64)))
    return (t / rms).astype(np.float32)


def outlier_channels(K: int, frac: float, seed: int) -> np.ndarray:
    """A seeded set of round(frac*K) (at least 1) distinct K-channel indices."""
    n = max(1, int(round(frac * K)))
    return np.sort(_rng(seed).choice(K, size=n, replace=False))


def scale_channels(x: np.ndarray, channels: np.ndarray, factor: float) -> np.ndarray:
    x[:, channels] *= np.float32(factor)
    return x


def group_spikes(x: np.ndarray, group: int, seed: int, value: float = 1000.0,
                 row_period: int = 8, row_phase: int = 3) -> np.ndarray:
    """In rows m % row_period == row_phase put one +-value per group of `group`
    columns, at a seeded position with a seeded sign."""
    M, K = x.shape
    rows = np.arange(row_phase, M, row_period)
    if rows.size == 0:
        return x
    G = K // group
    rng = _rng(seed)
    pos = rng.integers(0, group, size=(rows.size, G))
    sign = np.where(rng.integers(0, 2, size=(rows.size, G)) == 0, -1.0, 1.0).astype(np.float32)
    cols = np.arange(G)[None, :] * group + pos
    x[rows[:, None], cols] = sign * np.float32(value)
    return x


# ------------------------------------------------------------ workloads --

def act_small(M: int, K: int, seed: int = SEED_ACT) -> np.ndarray:
    return f32_to_bf16_bits(normal((M, K), seed))


def act_decode(M: int, K: int, seed: int = SEED_ACT) -> np.ndarray:
    x = normal((M, K), seed)
    scale_channels(x, outlier_channels(K, 0.01, SEED_STRUCT), 30.0)
    return f32_to_bf16_bits(x)


def act_prefill(M: int, K: int, seed: int = SEED_ACT) -> np.ndarray:
    return f32_to_bf16_bits(student_t_unit_rms((M, K), seed))


def act_quant(M: int, K: int, group: int = 128, seed: int = SEED_ACT) -> np.ndarray:
    x = normal((M, K), seed)
    group_spikes(x, group, SEED_STRUCT)
    return f32_to_bf16_bits(x)


def act_full_grid(M: int, K: int, seed: int = SEED_ACT) -> np.ndarray:
    x = normal((M, K), seed)
    scale_channels(x, outlier_channels(K, 0.005, SEED_STRUCT), 50.0)
    return f32_to_bf16_bits(x)


def weight_f32(N: int, K: int, seed: int = SEED_WEIGHT) -> np.ndarray:
    return normal((N, K), seed, std=0.02)


def weight_bf16(N: int, K: int, seed: int = SEED_WEIGHT) -> np.ndarray:
    return f32_to_bf16_bits(weight_f32(N, K, seed))


# Benchmark-sized inputs (row-blocked parallel draws, see normal_blocked).

def weight_bf16_blocked(N: int, K: int, seed: int = SEED_WEIGHT) -> np.ndarray:
    return f32_to_bf16_bits_par(normal_blocked((N, K), seed, std=0.02))


def act_full_grid_blocked(M: int, K: int, seed: int = SEED_ACT) -> np.ndarray:
    x = normal_blocked((M, K), seed)
    scale_channels(x, outlier_channels(K, 0.005, SEED_STRUCT), 50.0)
    return f32_to_bf16_bits_par(x)


def act_decode_blocked(M: int, K: int, seed: int = SEED_ACT) -> np.ndarray:
    x = normal_blocked((M, K), seed)
    scale_channels(x, outlier_channels(K, 0.01, SEED_STRUCT), 30.0)
    return f32_to_bf16_bits_par(x)


def act_prefill_blocked(M: int, K: int, seed: int = SEED_ACT, nu: float = 3.0,
                        block_rows: int = 1024) -> np.ndarray:
    """Student-t(nu) rows drawn per row block (stream SeedSequence([seed, b])),
    scaled to unit empirical RMS over the whole matrix (fp64)."""
    t = np.empty((M, K), dtype=np.float64)

    def fill(item):
        b, rows = item
        t[rows] = np.random.default_rng([seed, b]).standard_t(nu, size=t[rows].shape)

    blocks = _row_blocks((M, K), block_rows)
    _par_map(fill, blocks)
    rms = np.sqrt(np.mean(np.square(t)))
    x = np.empty((M, K), dtype=np.float32)

    def norm(item):
        _, rows = item
        x[rows] = t[rows] / rms

    _par_map(norm, blocks)
    return f32_to_bf16_bits_par(x)


def act_quant_blocked(M: int, K: int, group: int = 128, seed: int = SEED_ACT) -> np.ndarray:
    x = normal_blocked((M, K), seed)
    group_spikes(x, group, SEED_STRUCT)
    return f32_to_bf16_bits_par(x)


# The pages' M grid ("vLLM 量化 Kernel 配置机制" §2) and the workload shape sets.
M_GRID = (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128, 256, 512, 1024, 1536, 2048, 3072, 4096)
DECODE_M = (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128)
DECODE_NK = ((7168, 18432), (18432, 7168), (4096, 7168))
PREFILL_M = (256, 512, 1024, 1536, 2048, 3072, 4096)
PREFILL_NK = ((24576, 7168), (4096, 7168), (7168, 18432))
QUANT_M = (1, 64, 1024, 4096, 16384)
QUANT_K = (1536, 7168, 18432)
FULL_NK = ((1536, 7168), (7168, 1536), (4096, 7168), (7168, 18432), (18432, 7168), (24576, 7168))


# Grouped (MoE) workload: DeepSeek-V3 routed-expert projections (hidden 7168,
# expert width 2048: gate+up N=4096 K=7168, down N=7168 K=2048), 256 routed
# experts with top-8 routing, 32 of them on this GPU.
MOE_NK = ((4096, 7168), (7168, 2048))
MOE_E_TOTAL = 256
MOE_E_LOCAL = 32
MOE_TOP_K = 8
MOE_TOKENS = (128, 4096)  # decode batch, prefill chunk


def moe_counts(E: int, tokens: int, E_total: int = MOE_E_TOTAL, top_k: int = MOE_TOP_K,
               seed: int = SEED_STRUCT) -> np.ndarray:
    """Tokens routed to each of the first E experts (int32 [E]) when `tokens`
    tokens each pick top_k distinct experts of E_total, drawn with a seeded
    popularity vector (Dirichlet(0.5))."""
    g = _rng(seed)
    pop = g.dirichlet(np.full(E_total, 0.5))
    hits = np.zeros(E_total, dtype=np.int64)
    for _ in range(tokens):
        hits[g.choice(E_total, size=top_k, replace=False, p=pop)] += 1
    return hits[:E].astype(np.int32)


def moe_act(E: int, M_max: int, K: int, seed: int = SEED_ACT) -> np.ndarray:
    """Token rows of E experts, M_max rows each (bf16 bits [E*M_max, K])."""
    return act_decode(E * M_max, K, seed=seed)


def moe_weight_bf16(E: int, N: int, K: int, seed: int = SEED_WEIGHT) -> np.ndarray:
    """E stacked expert weights (bf16 bits [E, N, K]), expert e seeded seed+e."""
    return np.stack([weight_bf16(N, K, seed=seed + 1000 * e) for e in range(E)])
