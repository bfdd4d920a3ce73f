"""Shared helpers of the GPU parity tests: host<->device marshalling, oracle
evaluation over row samples, and the acceptance bounds.

Acceptance (the method's stated bar):
  * quantisation: codes and scales bit-exact;
  * GEMM, bf16/fp16 output: |gpu - ref| <= 2^-7 |ref| + 1e-4 max|ref| per element,
    with ref the unrounded fp64 oracle value;
  * GEMM, fp32 output: ||gpu - ref||_F / ||ref||_F <= 1e-5.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from block_scaled_fp8_group_gb300 import synth

TORCH_OUT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def to_dev_bits(bits: np.ndarray, dtype=torch.bfloat16) -> torch.Tensor:
    """uint16 bit patterns -> CUDA bf16/fp16 tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(dtype).cuda()


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def scales_to_dev(s: np.ndarray) -> torch.Tensor:
    if s.dtype == np.uint32:
        return torch.from_numpy(s.view(np.int32)).cuda()
    return torch.from_numpy(s).cuda()


def scales_bits(s) -> np.ndarray:
    a = s.cpu().numpy() if isinstance(s, torch.Tensor) else s
    return np.ascontiguousarray(a).view(np.uint32)


def oracle_rows(qa, sa, qw, sw, ue, rows, threads=16):
    """fp64 oracle values of the listed rows (all N columns), computed in
    parallel threads (the C oracle releases the GIL)."""
    rows = list(rows)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda m: oracle.gemm(qa, sa, qw, sw, ue, rows=(m, 1)), rows))
    return np.concatenate(parts, axis=0)


def oracle_full(qa, sa, qw, sw, ue, threads=16):
    M = qa.shape[0]
    chunk = max(1, (M + threads - 1) // threads)
    starts = list(range(0, M, chunk))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(
            lambda r0: oracle.gemm(qa, sa, qw, sw, ue, rows=(r0, min(chunk, M - r0))), starts))
    return np.concatenate(parts, axis=0)


def check_gemm(got: np.ndarray, ref: np.ndarray, out: str, what: str = ""):
    got = got.astype(np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if out in ("bf16", "fp16"):
        bound = 2.0 ** -7 * np.abs(ref) + 1e-4 * np.abs(ref).max()
        err = np.abs(got - ref)
        bad = err > bound
        if bad.any():
            i = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: {bad.sum()} elements out of bound; first {tuple(i)}: "
                                 f"got {got[tuple(i)]} ref {ref[tuple(i)]} bound {bound[tuple(i)]}")
    else:
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= 1e-5, f"{what}: relative Frobenius error {rel:.3e} > 1e-5"


def quantised_problem(M, N, K, ue, act_maker, weight="f32"):
    """Host-side inputs quantised by the oracle: (qa, sa, qw, sw)."""
    xb = act_maker(M, K)
    if weight == "f32":
        qw, sw = oracle.quant_weight(synth.weight_f32(N, K), oracle.FP32, 128, 128, ue)
    else:
        qw, sw = oracle.quant_weight(synth.weight_bf16(N, K), oracle.BF16, 128, 128, ue)
    qa, sa = oracle.quant_act(xb, oracle.BF16, 128, ue)
    return xb, qa, sa, qw, sw


def sample_rows(M: int, k: int = 8, seed: int = 11):
    """Rows 0, M-1, the first and last row of the second 128-row tile, the
    first row of the last 128-row tile and a seeded sample of the rest."""
    base = {0, M - 1, (M - 1) // 128 * 128}
    if M > 128:
        base |= {127, 128, min(M - 1, 255)}
    rng = np.random.default_rng(seed)
    extra = rng.choice(M, size=min(M, k), replace=False)
    return sorted(base | set(int(e) for e in extra))
