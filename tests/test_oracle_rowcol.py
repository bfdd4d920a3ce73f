"""Pins of the oracle's per-token x per-channel formats (FP8_Dynamic and
W8A8_INT8 of "用 Helion 为 vLLM 构建高性能可移植线性后端", 范围).

Quant:
* A row of 128 elements is one 1x128 group: the e4m3 per-row quant equals the
  (separately pinned) per-token-group quant with group 128, and a weight's
  per-channel quant equals the 128x128 block quant with a 1 x K block.
* int8: every code is a nearest integer to x/s (|q*s - x| <= s/2 up to the
  fp32 division's rounding), exact halves go to the even neighbour, the amax
  element maps to +-127, |q| <= 127, all-zero rows give the eps scale.
* Sign symmetry and power-of-two scaling of a row.
GEMM:
* Exact rational brute force on tiny inputs (correctly rounded: bit-equal).
* Equal to the (pinned) block-scaled GEMM when the scales are constant along
  the row's groups and within each 128-row weight block.
* int8 sums against numpy's int64 matmul; identity weights in closed form.
A transposed operand, a scale taken from the wrong side, a dropped scale, a
sign error or a wrong rounding rule each fails at least one of these.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_scaled_fp8_group_gb300 import synth

DEC = oracle.e4m3_decode_all()


def f32_from_bf16(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------- quant --

@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_rows_e4m3_equals_group_quant_at_k128(dt):
    xb = synth.act_quant(64, 128)
    if dt == "fp16":
        xb = synth.f32_to_f16_bits(f32_from_bf16(xb))
    code = oracle.BF16 if dt == "bf16" else oracle.FP16
    q, s = oracle.quant_rows(xb, code)
    qg, sg = oracle.quant_act(xb, code, 128, False)
    assert np.array_equal(q, qg)
    assert np.array_equal(s, sg[0, :64])


def test_rows_e4m3_equals_one_by_k_weight_block():
    w = synth.weight_f32(70, 512)
    q, s = oracle.quant_rows(w, oracle.FP32)
    qb, sb = oracle.quant_weight(w, oracle.FP32, 1, 512, False)
    assert np.array_equal(q, qb)
    assert np.array_equal(s, sb[:, 0])


@pytest.mark.parametrize("int8", [False, True])
def test_rows_amax_maps_to_max_code(int8):
    xb = synth.act_decode(16, 1024)
    x = f32_from_bf16(xb)
    q, s = oracle.quant_rows(xb, oracle.BF16, int8=int8)
    for r in range(16):
        i = int(np.argmax(np.abs(x[r])))
        if int8:
            assert abs(int(q[r, i])) == 127
            assert int(q[r, i]) * np.sign(x[r, i]) > 0
        else:
            assert q[r, i] in (0x7E, 0xFE)
        if int8:
            assert np.all(np.abs(q[r].astype(np.int32)) <= 127)
        else:
            assert np.all((q[r] & 0x7F) <= 0x7E)


def test_rows_int8_nearest_integer():
    """|q - x/s| <= 1/2 + (rounding of the fp32 quotient), for every element."""
    for xb in (synth.act_decode(8, 2048), synth.act_prefill(8, 2048)):
        x = f32_from_bf16(xb).astype(np.float64)
        q, s = oracle.quant_rows(xb, oracle.BF16, int8=True)
        ratio = x / s.astype(np.float64)[:, None]
        # fp32 division: |fp32(x/s) - x/s| <= 2^-24 * 128
        assert np.all(np.abs(q.astype(np.float64) - ratio) <= 0.5 + 2.0 ** -17)


def test_rows_int8_ties_to_even():
    # amax = 127 * 2^-3 makes s = 2^-3 exactly; x = (k + 1/2) * 2^-3 is an
    # exact half (bf16: 2k+1 <= 255 fits its 8-bit significand)
    k = np.arange(-127, 127)
    vals = np.concatenate([[127 * 0.125], (k + 0.5) * 0.125]).astype(np.float32)
    xb = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(f32_from_bf16(xb), vals)  # representable
    K = (len(vals) + 15) // 16 * 16
    row = np.zeros(K, dtype=np.uint16)
    row[:len(vals)] = xb
    q, s = oracle.quant_rows(row[None, :], oracle.BF16, int8=True)
    assert s[0] == np.float32(0.125)
    got = q[0, 1:len(vals)].astype(np.int64)
    lo, hi = k, k + 1
    want = np.where(lo % 2 == 0, lo, hi)
    assert np.array_equal(got, want)


def test_rows_e4m3_ties_to_even():
    # amax = 448 * 2^-4 gives s = 2^-4; x = midpoint of two adjacent e4m3
    # values (times s) must take the code with the even mantissa
    finite = np.array([DEC[c] for c in range(0x7F)])  # 0 .. 448, increasing
    mids = (finite[1:] + finite[:-1]) / 2
    vals = np.concatenate([[448.0], mids]) * 2.0 ** -4
    vals32 = vals.astype(np.float32)
    assert np.array_equal(vals32.astype(np.float64), vals)
    # fp32 inputs hold every midpoint exactly
    q, s = oracle.quant_rows(vals32[None, :], oracle.FP32)
    assert s[0] == np.float32(2.0 ** -4)
    for i, c in enumerate(q[0, 1:]):
        assert c in (i, i + 1) and c % 2 == 0, (i, c)


@pytest.mark.parametrize("int8", [False, True])
def test_rows_zero_row_and_symmetry(int8):
    xb = synth.act_decode(4, 512)
    xb[2] = 0
    q, s = oracle.quant_rows(xb, oracle.BF16, int8=int8)
    eps = np.float32(1e-10) / np.float32(127.0 if int8 else 448.0)
    assert s[2] == eps and np.all(q[2] == 0)
    qn, sn = oracle.quant_rows(xb ^ np.uint16(0x8000), oracle.BF16, int8=int8)
    assert np.array_equal(sn, s)
    if int8:
        assert np.array_equal(qn.astype(np.int32), -q.astype(np.int32))
    else:
        nz = (q & 0x7F) != 0
        assert np.array_equal(qn[nz], q[nz] ^ 0x80)


@pytest.mark.parametrize("int8", [False, True])
def test_rows_power_of_two_scaling(int8):
    x = synth.weight_f32(6, 384)
    q, s = oracle.quant_rows(x, oracle.FP32, int8=int8)
    q2, s2 = oracle.quant_rows((x * np.float32(2.0 ** 5)).astype(np.float32), oracle.FP32,
                               int8=int8)
    assert np.array_equal(q2, q)
    assert np.array_equal(s2, s * np.float32(2.0 ** 5))


# -------------------------------------------------------------------- GEMM --

def val(code, int8):
    return Fraction(int(np.int8(code))) if int8 else Fraction(DEC[code])


@pytest.mark.parametrize("int8", [False, True])
def test_gemm_exact_rational(int8):
    M, N, K = 3, 5, 256
    qa, sa = oracle.quant_rows(synth.act_decode(M, K), oracle.BF16, int8=int8)
    qw, sw = oracle.quant_rows(synth.weight_f32(N, K), oracle.FP32, int8=int8)
    ref = oracle.gemm_rowcol(qa, sa, qw, sw, int8)
    ua, uw = qa.view(np.uint8), qw.view(np.uint8)
    for m in range(M):
        for n in range(N):
            S = sum(val(ua[m, k], int8) * val(uw[n, k], int8) for k in range(K))
            exact = Fraction(float(sa[m])) * Fraction(float(sw[n])) * S
            # sa*sw is exact and S is exact: one rounding, to nearest
            assert ref[m, n] == float(exact), (m, n)


def test_gemm_e4m3_equals_block_gemm_with_constant_scales():
    M, N, K = 7, 256, 512
    qa, sa = oracle.quant_rows(synth.act_decode(M, K), oracle.BF16)
    qw, _ = oracle.quant_rows(synth.weight_f32(N, K), oracle.FP32)
    sw = np.repeat(np.array([0.0123, 0.5], dtype=np.float32), 128)  # constant per 128 rows
    ref = oracle.gemm_rowcol(qa, sa, qw, sw)
    G, Mp = K // 128, (M + 3) // 4 * 4
    sa_blk = np.zeros((G, Mp), dtype=np.float32)
    sa_blk[:, :M] = sa[None, :]
    sw_blk = np.repeat(np.array([[0.0123], [0.5]], dtype=np.float32), G, axis=1)
    blk = oracle.gemm(qa, sa_blk, qw, sw_blk, False)
    assert np.allclose(ref, blk, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gemm_int8_sum_against_numpy():
    M, N, K = 9, 130, 1536
    qa, sa = oracle.quant_rows(synth.act_prefill(M, K), oracle.BF16, int8=True)
    qw, sw = oracle.quant_rows(synth.weight_f32(N, K), oracle.FP32, int8=True)
    ref = oracle.gemm_rowcol(qa, sa, qw, sw, True)
    S = qa.astype(np.int64) @ qw.astype(np.int64).T
    scale = sa.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    assert np.array_equal(ref, scale * S.astype(np.float64))


@pytest.mark.parametrize("int8", [False, True])
def test_gemm_identity_weights(int8):
    K = 256
    qa, sa = oracle.quant_rows(synth.act_decode(4, K), oracle.BF16, int8=int8)
    w = np.eye(K, dtype=np.float32)
    qw, sw = oracle.quant_rows(w, oracle.FP32, int8=int8)
    # every weight row has amax 1: s = fp32(1/127) or fp32(1/448); the 1.0
    # quantises to the largest code (127, or 448 = 0x7E)
    top = 127.0 if int8 else 448.0
    assert np.all(sw == np.float32(1.0) / np.float32(top))
    ref = oracle.gemm_rowcol(qa, sa, qw, sw, int8)
    aval = qa.astype(np.float64) if int8 else DEC[qa]
    want = (sa.astype(np.float64)[:, None] * float(sw[0])) * (aval * top)
    assert np.array_equal(ref, want)
