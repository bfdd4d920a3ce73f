"""Pins of the oracle's block-scaled GEMM (fp64).

* Brute force in exact rational arithmetic (fractions.Fraction) on tiny inputs.
* Dequantise-then-matmul with numpy's fp64 matmul (a library routine).
* Identity and all-ones weights, whose results have closed forms.
* Single-slab (K = 128) and 1x1 special cases, element accessor = full GEMM.
* calc_diff special cases.
A transposed operand, a wrong scale index (row vs column block, K block), a
dropped scale or a sign error each fails at least one of these.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_scaled_fp8_group_gb300 import synth

DEC = oracle.e4m3_decode_all()


def quantised_problem(M, N, K, ue, act=synth.act_decode, seed=0):
    xb = act(M, K, seed=seed)
    w = synth.weight_f32(N, K, seed=seed + 1)
    qa, sa = oracle.quant_act(xb, oracle.BF16, 128, ue)
    qw, sw = oracle.quant_weight(w, oracle.FP32, 128, 128, ue)
    return qa, sa, qw, sw


def act_scales_dense(sa, ue, M, K):
    G = K // 128
    return np.array([[oracle.act_scale(sa, ue, M, K, 128, m, g) for g in range(G)]
                     for m in range(M)])


@pytest.mark.parametrize("ue", [False, True])
def test_exact_rational_brute_force(ue):
    M, N, K = 3, 130, 256  # partial weight row block (rows 128, 129)
    qa, sa, qw, sw = quantised_problem(M, N, K, ue)
    ref = oracle.gemm(qa, sa, qw, sw, ue)
    sa_d = act_scales_dense(sa, ue, M, K)
    G = K // 128
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            mag = Fraction(0)
            for kb in range(G):
                slab = sum(Fraction(DEC[qa[m, k]]) * Fraction(DEC[qw[n, k]])
                           for k in range(kb * 128, (kb + 1) * 128))
                term = Fraction(sa_d[m, kb]) * Fraction(float(sw[n // 128, kb])) * slab
                exact += term
                mag += abs(term)
            err = abs(Fraction(ref[m, n]) - exact)
            assert err <= mag * Fraction(4 * G, 2 ** 53), (m, n)


@pytest.mark.parametrize("ue", [False, True])
def test_dequantise_then_matmul(ue):
    M, N, K = 9, 384, 1024
    qa, sa, qw, sw = quantised_problem(M, N, K, ue, act=synth.act_prefill)
    ref = oracle.gemm(qa, sa, qw, sw, ue)
    a_deq = DEC[qa] * np.repeat(act_scales_dense(sa, ue, M, K), 128, axis=1)
    w_deq = DEC[qw] * np.repeat(np.repeat(sw.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    lib = a_deq @ w_deq.T
    bound = np.abs(a_deq) @ np.abs(w_deq).T
    assert np.all(np.abs(ref - lib) <= 1e-12 * bound + 1e-300)
    # and the result is not trivially zero
    assert np.abs(ref).max() > 0.1


def test_identity_weights_ue8m0_closed_form():
    M, K = 5, 256
    xb = synth.act_decode(M, K)
    qa, sa = oracle.quant_act(xb, oracle.BF16, 128, True)
    qw, sw = oracle.quant_weight(np.eye(K, dtype=np.float32), oracle.FP32, 128, 128, True)
    # diagonal blocks: amax 1 -> s = 2^-8, 1/s = 256 -> code 0x78 -> dequant exactly 1
    assert np.all(sw[[0, 1], [0, 1]] == 2.0 ** -8)
    assert np.all(np.diag(qw) == 0x78) and np.all(qw[~np.eye(K, dtype=bool)] == 0)
    ref = oracle.gemm(qa, sa, qw, sw, True)
    want = DEC[qa] * np.repeat(act_scales_dense(sa, True, M, K), 128, axis=1)
    np.testing.assert_array_equal(ref, want)


def test_identity_weights_fp32_closed_form():
    M, K = 4, 384
    xb = synth.act_small(M, K)
    qa, sa = oracle.quant_act(xb, oracle.BF16, 128, False)
    qw, sw = oracle.quant_weight(np.eye(K, dtype=np.float32), oracle.FP32, 128, 128, False)
    s = np.float32(1.0) / np.float32(448.0)
    assert np.all(np.diag(sw) == s) and np.all(np.diag(qw) == 0x7E)
    ref = oracle.gemm(qa, sa, qw, sw, False)
    want = (DEC[qa] * 448.0) * (np.repeat(act_scales_dense(sa, False, M, K), 128, axis=1)
                                * float(s))
    np.testing.assert_allclose(ref, want, rtol=1e-15, atol=0)


@pytest.mark.parametrize("ue", [False, True])
def test_all_ones_weights(ue):
    M, N, K = 6, 256, 512
    xb = synth.act_prefill(M, K)
    qa, sa = oracle.quant_act(xb, oracle.BF16, 128, ue)
    qw, sw = oracle.quant_weight(np.ones((N, K), dtype=np.float32), oracle.FP32, 128, 128, ue)
    c = 1.0 if ue else 448.0 * float(np.float32(1) / np.float32(448))
    ref = oracle.gemm(qa, sa, qw, sw, ue)
    rowsum = (DEC[qa] * np.repeat(act_scales_dense(sa, ue, M, K), 128, axis=1)).sum(axis=1)
    for n in range(N):
        np.testing.assert_allclose(ref[:, n], rowsum * c, rtol=1e-13)
    # all columns identical
    assert np.all(ref == ref[:, :1])


def test_single_slab_and_one_by_one():
    for M, N, K in ((1, 1, 128), (1, 128, 128), (2, 3, 128)):
        qa, sa, qw, sw = quantised_problem(M, N, K, False, act=synth.act_small)
        ref = oracle.gemm(qa, sa, qw, sw, False)
        for m in range(M):
            for n in range(N):
                slab = float(np.dot(DEC[qa[m]], DEC[qw[n]]))
                want = slab * (float(sa[0, m]) * float(sw[n // 128, 0]))
                assert ref[m, n] == want


def test_row_slices_and_elements_agree_with_full():
    M, N, K = 7, 256, 640
    qa, sa, qw, sw = quantised_problem(M, N, K, True)
    full = oracle.gemm(qa, sa, qw, sw, True)
    part = oracle.gemm(qa, sa, qw, sw, True, rows=(3, 4))
    np.testing.assert_array_equal(part, full[3:7])
    for m, n in ((0, 0), (6, 255), (3, 129)):
        assert oracle.gemm_elem(qa, sa, qw, sw, True, m, n) == full[m, n]


def test_swapping_operands_changes_result():
    # guards against a transposed operand: A@W^T differs from W@A^T layouts
    M, N, K = 128, 128, 256
    qa, sa, qw, sw = quantised_problem(M, N, K, False)
    ref = oracle.gemm(qa, sa, qw, sw, False)
    a_deq = DEC[qa] * np.repeat(act_scales_dense(sa, False, M, K), 128, axis=1)
    w_deq = DEC[qw] * np.repeat(np.repeat(sw.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    assert not np.allclose(ref, (w_deq @ a_deq.T), rtol=1e-3)
    np.testing.assert_allclose(ref, a_deq @ w_deq.T, rtol=1e-10, atol=1e-12)


def test_calc_diff_special_cases():
    x = synth.normal((1000,), seed=5).astype(np.float64)
    assert oracle.calc_diff(x, x) == 0.0
    assert oracle.calc_diff(x, -x) == 2.0
    assert oracle.calc_diff(x, np.zeros_like(x)) == 1.0
    # scale by a factor a: 1 - 2a/(1+a^2)
    a = 1.5
    np.testing.assert_allclose(oracle.calc_diff(x, a * x), 1 - 2 * a / (1 + a * a), rtol=1e-14)
