"""Pins of the oracle's block INT8 format (int8_w8a8 with block_shape
[128,128] of "vLLM 量化 Kernel 配置机制" §1).

* One group per row (group = K) is the pinned per-row int8 quant; a 1 x K
  weight block is the pinned per-channel int8 quant.
* Every code is a nearest integer to x / s of its own group; the group amax
  maps to +-127; all-zero groups take the eps scale.
* GEMM: exact rational brute force; with one K slab (K = 128) and constant
  scales per row / per 128-row block it equals the pinned rowwise int8 GEMM;
  per-slab integer sums against numpy's int64 matmul.
A wrong group index, a scale from the wrong slab or block, or a sum over the
wrong K range fails at least one of these.
"""
from fractions import Fraction

import numpy as np

import oracle
from block_scaled_fp8_group_gb300 import synth


def f32_of_bf16(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def test_one_group_per_row_is_the_rowwise_quant():
    xb = synth.act_decode(9, 512)
    q, s = oracle.quant_act_int8(xb, oracle.BF16, group=512)
    qr, sr = oracle.quant_rows(xb, oracle.BF16, int8=True)
    assert np.array_equal(q, qr)
    assert np.array_equal(s[0, :9], sr)
    assert np.all(s[0, 9:] == 0)  # padding rows


def test_one_by_k_weight_block_is_the_per_channel_quant():
    w = synth.weight_f32(40, 384)
    q, s = oracle.quant_weight_int8(w, oracle.FP32, 1, 384)
    qr, sr = oracle.quant_rows(w, oracle.FP32, int8=True)
    assert np.array_equal(q, qr)
    assert np.array_equal(s[:, 0], sr)


def test_codes_nearest_and_amax_per_group():
    xb = synth.act_quant(16, 1024)  # rows with +-1000 spikes per group
    x = f32_of_bf16(xb).astype(np.float64)
    q, s = oracle.quant_act_int8(xb, oracle.BF16)
    G = 1024 // 128
    for m in range(16):
        for g in range(G):
            xs = x[m, g * 128:(g + 1) * 128]
            qs = q[m, g * 128:(g + 1) * 128].astype(np.float64)
            sc = float(s[g, m])
            assert np.all(np.abs(qs - xs / sc) <= 0.5 + 2.0 ** -17)
            i = int(np.argmax(np.abs(xs)))
            assert abs(qs[i]) == 127
    xb[3, 128:256] = 0
    q, s = oracle.quant_act_int8(xb, oracle.BF16)
    assert s[1, 3] == np.float32(1e-10) / np.float32(127.0)
    assert np.all(q[3, 128:256] == 0)


def test_weight_blocks_take_their_own_amax():
    w = synth.weight_f32(200, 256)  # a partial last row block (rows 128..199)
    q, s = oracle.quant_weight_int8(w, oracle.FP32)
    for nb in range(2):
        for kb in range(2):
            blk = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = np.float32(np.abs(blk).max())
            assert s[nb, kb] == amax / np.float32(127.0)
            qb = q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            assert np.abs(qb).max() == 127


def test_gemm_exact_rational():
    M, N, K = 3, 130, 256
    qa, sa = oracle.quant_act_int8(synth.act_decode(M, K), oracle.BF16)
    qw, sw = oracle.quant_weight_int8(synth.weight_f32(N, K), oracle.FP32)
    ref = oracle.gemm_int8_block(qa, sa, qw, sw)
    for m in range(M):
        for n in (0, 1, 127, 128, 129):
            exact, mag = Fraction(0), Fraction(0)
            for kb in range(2):
                S = sum(int(qa[m, k]) * int(qw[n, k]) for k in range(kb * 128, (kb + 1) * 128))
                t = Fraction(float(sa[kb, m])) * Fraction(float(sw[n // 128, kb])) * S
                exact += t
                mag += abs(t)
            assert abs(Fraction(ref[m, n]) - exact) <= mag * Fraction(8, 2 ** 53), (m, n)


def test_gemm_single_slab_equals_rowwise():
    M, N, K = 5, 256, 128
    xb = synth.act_decode(M, K)
    qa, sa = oracle.quant_act_int8(xb, oracle.BF16)
    qw, sw = oracle.quant_weight_int8(synth.weight_f32(N, K), oracle.FP32)
    ref = oracle.gemm_int8_block(qa, sa, qw, sw)
    # one slab: sa is one scale per row, sw one per 128-row block
    rr = oracle.gemm_rowcol(qa, sa[0, :M].copy(), qw, np.repeat(sw[:, 0], 128).copy(), True)
    assert np.array_equal(ref, rr)


def test_gemm_slab_sums_against_numpy():
    M, N, K = 6, 256, 512
    qa, sa = oracle.quant_act_int8(synth.act_prefill(M, K), oracle.BF16)
    qw, sw = oracle.quant_weight_int8(synth.weight_f32(N, K), oracle.FP32)
    ref = oracle.gemm_int8_block(qa, sa, qw, sw)
    want = np.zeros((M, N))
    for kb in range(K // 128):
        S = qa[:, kb * 128:(kb + 1) * 128].astype(np.int64) @ \
            qw[:, kb * 128:(kb + 1) * 128].astype(np.int64).T
        f = sa[kb, :M].astype(np.float64)[:, None] * \
            np.repeat(sw[:, kb].astype(np.float64), 128)[None, :N]
        want = want + f * S
    assert np.allclose(ref, want, rtol=1e-13, atol=1e-13 * np.abs(want).max())
