"""Pins of the oracle's grouped (MoE) GEMM, masked layout.

* Dequantise-then-matmul per expert with numpy's fp64 matmul (a library
  routine; the dequantisation is written here from the e4m3 decode table and
  the scale layouts, not through the oracle's GEMM).
* Counts are clamped to [0, M_max]; rows past an expert's count keep the
  caller's values.
* Permuting the experts (their weights, token rows and counts together)
  permutes the output blocks.
A wrong expert offset for the weights, scales or token rows, a count that is
not clamped, or rows written past a count each fails at least one of these.
"""
import numpy as np
import pytest

import oracle
from block_scaled_fp8_group_gb300 import synth

DEC = oracle.e4m3_decode_all()


def grouped_problem(E, M_max, N, K, ue, seed=0):
    xb = synth.moe_act(E, M_max, K, seed=seed)
    qa, sa = oracle.quant_act(xb, oracle.BF16, 128, ue)
    wb = synth.moe_weight_bf16(E, N, K, seed=seed + 1)
    qs = [oracle.quant_weight(wb[e], oracle.BF16, 128, 128, ue) for e in range(E)]
    qw = np.stack([q for q, _ in qs])
    sw = np.stack([s for _, s in qs])
    return xb, qa, sa, qw, sw


def act_scale_matrix(sa, ue, rows, K):
    """[rows, G] activation scales read from the column-major layout."""
    G = K // 128
    Mp = (rows + 3) // 4 * 4
    if ue:
        words = sa.reshape(-1)[: ((G + 3) // 4) * Mp].reshape((G + 3) // 4, Mp)
        out = np.empty((rows, G))
        for g in range(G):
            byte = (words[g // 4, :rows].astype(np.uint32) >> (8 * (g % 4))) & 0xFF
            out[:, g] = np.ldexp(1.0, byte.astype(np.int64) - 127)
        return out
    return sa.reshape(-1)[: G * Mp].reshape(G, Mp)[:, :rows].T.astype(np.float64)


@pytest.mark.parametrize("ue", [False, True])
def test_grouped_dequantise_then_matmul(ue):
    E, M_max, N, K = 4, 8, 256, 512
    counts = np.array([3, 0, 8, 5], dtype=np.int32)
    _, qa, sa, qw, sw = grouped_problem(E, M_max, N, K, ue)
    ref = oracle.grouped_gemm(qa, sa, qw, sw, counts, ue)
    a_deq = DEC[qa] * np.repeat(act_scale_matrix(sa, ue, E * M_max, K), 128, axis=1)
    for e in range(E):
        w_deq = DEC[qw[e]] * np.repeat(np.repeat(sw[e].astype(np.float64), 128, axis=0)[:N],
                                       128, axis=1)
        rows = slice(e * M_max, e * M_max + counts[e])
        lib = a_deq[rows] @ w_deq.T
        bound = np.abs(a_deq[rows]) @ np.abs(w_deq).T
        assert np.all(np.abs(ref[rows] - lib) <= 1e-12 * bound + 1e-300), e
        assert counts[e] == 0 or np.abs(lib).max() > 0.01
        # rows past the count are not written (NaN when no output is given)
        assert np.all(np.isnan(ref[e * M_max + counts[e]:(e + 1) * M_max]))


def test_grouped_counts_clamped_and_rows_kept():
    E, M_max, N, K = 3, 4, 128, 256
    _, qa, sa, qw, sw = grouped_problem(E, M_max, N, K, True)
    base = np.full((E * M_max, N), 7.0)
    over = oracle.grouped_gemm(qa, sa, qw, sw, np.array([99, -5, 2]), True, out=base.copy())
    full = oracle.grouped_gemm(qa, sa, qw, sw, np.array([4, 0, 2]), True, out=base.copy())
    assert np.array_equal(over, full)
    assert np.all(full[4:8] == 7.0) and np.all(full[10:12] == 7.0)
    assert not np.any(full[0:4] == 7.0)


def test_grouped_expert_permutation():
    E, M_max, N, K = 3, 4, 128, 256
    counts = np.array([4, 2, 3], dtype=np.int32)
    xb, qa, sa, qw, sw = grouped_problem(E, M_max, N, K, False)
    ref = oracle.grouped_gemm(qa, sa, qw, sw, counts, False)
    perm = [2, 0, 1]
    xb_p = np.concatenate([xb[e * M_max:(e + 1) * M_max] for e in perm])
    qa_p, sa_p = oracle.quant_act(xb_p, oracle.BF16, 128, False)
    ref_p = oracle.grouped_gemm(qa_p, sa_p, qw[perm], sw[perm], counts[perm], False)
    for i, e in enumerate(perm):
        assert np.array_equal(ref_p[i * M_max:(i + 1) * M_max], ref[e * M_max:(e + 1) * M_max],
                              equal_nan=True)
