"""Pins of the oracle's activation and weight quantisation.

Checked against: hand-derived closed forms (tests/golden/act_quant_tiny.txt),
the invariants the method fixes (|q| <= 448, amax -> +-448 with fp32 scales,
power-of-two scales in (amax/448, 2*amax/448] with UE8M0), symmetry and
power-of-two equivariance, the all-zero group, the spike example, and an
independent re-implementation on torch CPU ops (torch's float8_e4m3fn cast,
which rounds to nearest even for |y| <= 448).
"""
import math
import os
import re

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_group_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NAN_CODES = (0x7F, 0xFF)


def unpack_ue8m0(s_packed: np.ndarray, G: int) -> np.ndarray:
    """[ceil(G/4), Mp] uint32 -> [G, Mp] float64 scales 2^(byte-127) (0 for byte 0)."""
    Gq, Mp = s_packed.shape
    out = np.zeros((G, Mp))
    for g in range(G):
        byte = (s_packed[g // 4] >> np.uint32(8 * (g % 4))) & np.uint32(0xFF)
        out[g] = np.where(byte == 0, 0.0, np.exp2(byte.astype(np.float64) - 127))
    return out


def decode_codes(q):
    t = oracle.e4m3_decode_all()
    return t[q]


# ----------------------------------------------------------- golden tiny --

def read_golden_act_tiny():
    """Parses tests/golden/act_quant_tiny.txt (see its header)."""
    rows = {}
    with open(os.path.join(GOLDEN, "act_quant_tiny.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, _, val = line.partition("=")
            rows[key.strip()] = val.strip()
    return rows


def _golden_scale(tok: str) -> float:
    m = re.fullmatch(r"div\(([^,]+),([^)]+)\)", tok)
    if m:
        return float(np.float32(float(m.group(1))) / np.float32(float(m.group(2))))
    return float.fromhex(tok) if tok.startswith("0x") else float(tok)


def _golden_codes(spec: str, K: int) -> np.ndarray:
    want = np.zeros(K, dtype=np.uint8)
    for tok in spec.split():
        cols, _, code = tok.partition(":")
        lo, _, hi = cols.partition("-")
        want[int(lo):int(hi or lo) + 1] = int(code, 16)
    return want


def test_golden_act_quant_tiny():
    g = read_golden_act_tiny()
    M, K = 3, 512  # 3 rows, 4 groups of 128
    x = np.zeros((M, K), dtype=np.float32)
    for gi in range(4):  # row 0: one value 448*2^(g-2) at column 5 of group g
        x[0, gi * 128 + 5] = 448.0 * 2.0 ** (gi - 2)
    x[1, 0:128] = 1.0
    x[1, 128:256] = 0.25
    x[1, 128 + 7] = -3.5
    x[1, 384:512] = 1.0
    x[1, 384 + 100] = 1000.0
    for gi in range(4):  # row 2: constant groups 448*2^-g
        x[2, gi * 128:(gi + 1) * 128] = 448.0 * 2.0 ** (-gi)
    xb = synth.f32_to_bf16_bits(x)
    assert np.array_equal(synth.bf16_bits_to_f32(xb), x)  # all exact in bf16

    for mode, ue in (("fp32", False), ("ue8m0", True)):
        q, s = oracle.quant_act(xb, oracle.BF16, 128, ue)
        exp_s = np.array([_golden_scale(t) for t in g[f"{mode}.scales"].split()]).reshape(4, 4)
        got_s = unpack_ue8m0(s, 4) if ue else s.astype(np.float64)
        np.testing.assert_array_equal(got_s, exp_s, err_msg=mode)
        for r in range(3):
            want = _golden_codes(g[f"{mode}.row{r}.codes"], K)
            np.testing.assert_array_equal(q[r], want, err_msg=f"{mode} row {r}")


# ------------------------------------------------------------- invariants --

@pytest.fixture(scope="module")
def quant_data():
    M, K = 37, 1536  # ragged M (Mp = 40), G = 12
    return synth.act_quant(M, K), M, K


@pytest.mark.parametrize("ue", [False, True])
def test_invariants(quant_data, ue):
    xb, M, K = quant_data
    G = K // 128
    q, s = oracle.quant_act(xb, oracle.BF16, 128, ue)
    assert not np.isin(q, NAN_CODES).any()
    deq = np.abs(decode_codes(q))
    assert deq.max() <= 448.0
    x = synth.bf16_bits_to_f32(xb).astype(np.float64)
    amax = np.abs(x).reshape(M, G, 128).max(axis=2)
    sc = unpack_ue8m0(s, G) if ue else s.astype(np.float64)
    Mp = (M + 3) // 4 * 4
    assert sc.shape == (G, Mp)
    assert np.all(sc[:, M:] == 0), "padding rows must be zero"
    sc = sc[:, :M].T  # [M, G]
    if ue:
        mant, _ = np.frexp(sc)
        assert np.all(mant == 0.5), "UE8M0 scales must be powers of two"
        r = amax / sc
        assert np.all(r > 224.0) and np.all(r <= 448.0)
    else:
        # the amax element of each group maps to +-448
        idx = np.abs(x).reshape(M, G, 128).argmax(axis=2)
        codes = q.reshape(M, G, 128)[np.arange(M)[:, None], np.arange(G)[None, :], idx]
        assert np.all((codes & 0x7F) == 0x7E)
        np.testing.assert_allclose(sc, amax / 448.0, rtol=2 ** -23)


@pytest.mark.parametrize("ue", [False, True])
def test_negation_flips_sign_only(quant_data, ue):
    xb, M, K = quant_data
    q1, s1 = oracle.quant_act(xb, oracle.BF16, 128, ue)
    q2, s2 = oracle.quant_act(xb ^ np.uint16(0x8000), oracle.BF16, 128, ue)
    np.testing.assert_array_equal(s1, s2)
    np.testing.assert_array_equal(q2, q1 ^ np.uint8(0x80))


@pytest.mark.parametrize("ue", [False, True])
@pytest.mark.parametrize("j", [-3, 2, 5])
def test_power_of_two_equivariance(quant_data, ue, j):
    xb, M, K = quant_data
    x = synth.bf16_bits_to_f32(xb)
    xs = synth.f32_to_bf16_bits(x * np.float32(2.0 ** j))
    assert np.array_equal(synth.bf16_bits_to_f32(xs), x * np.float32(2.0 ** j))
    q1, s1 = oracle.quant_act(xb, oracle.BF16, 128, ue)
    q2, s2 = oracle.quant_act(xs, oracle.BF16, 128, ue)
    np.testing.assert_array_equal(q1, q2)
    G = K // 128
    a1 = unpack_ue8m0(s1, G) if ue else s1.astype(np.float64)
    a2 = unpack_ue8m0(s2, G) if ue else s2.astype(np.float64)
    np.testing.assert_array_equal(a2, a1 * 2.0 ** j)


def test_all_zero_group():
    xb = np.zeros((1, 256), dtype=np.uint16)
    eps_scale = np.float32(1e-10) / np.float32(448.0)
    q, s = oracle.quant_act(xb, oracle.BF16, 128, False)
    assert np.all(q == 0)
    assert s[0, 0] == eps_scale and s[1, 0] == eps_scale
    q, s = oracle.quant_act(xb, oracle.BF16, 128, True)
    assert np.all(q == 0)
    e = math.ceil(math.log2(float(eps_scale)))
    assert unpack_ue8m0(s, 2)[0, 0] == 2.0 ** e


def test_spike_worked_example():
    # a group holding +1000 and N(0,1) noise elsewhere
    x = synth.normal((1, 128), seed=7)
    x[0, 40] = 1000.0
    xb = synth.f32_to_bf16_bits(x)
    q, s = oracle.quant_act(xb, oracle.BF16, 128, True)
    assert unpack_ue8m0(s, 1)[0, 0] == 4.0  # 1000/448 = 2.23 -> 2^ceil(log2) = 4
    assert q[0, 40] == 0x78  # 1000/4 = 250 -> nearest e4m3 grid point is 256
    q, s = oracle.quant_act(xb, oracle.BF16, 128, False)
    assert s[0, 0] == np.float32(1000.0) / np.float32(448.0)
    assert q[0, 40] == 0x7E


def test_fp16_input_matches_bf16_path_on_shared_values():
    # values exactly representable in both formats quantise identically
    rng = np.random.default_rng(3)
    v = (rng.integers(-64, 64, size=(4, 256)) / 8.0).astype(np.float32)
    qa, sa = oracle.quant_act(synth.f32_to_bf16_bits(v), oracle.BF16, 128, False)
    qb, sb = oracle.quant_act(synth.f32_to_f16_bits(v), oracle.FP16, 128, False)
    np.testing.assert_array_equal(qa, qb)
    np.testing.assert_array_equal(sa, sb)


# ---------------------------------------------- independent torch version --

def torch_quant_act(x_f32: np.ndarray, ue: bool):
    x = torch.from_numpy(x_f32)
    M, K = x.shape
    g = x.view(M, K // 128, 128)
    amax = g.abs().amax(dim=2)
    s = torch.clamp(amax, min=torch.tensor(1e-10, dtype=torch.float32)) / 448.0
    if ue:
        s = torch.exp2(torch.ceil(torch.log2(s.double()))).float()
    y = torch.clamp(g / s[..., None], -448.0, 448.0)
    q = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(M, K)
    return q.numpy(), s.numpy()


@pytest.mark.parametrize("ue", [False, True])
@pytest.mark.parametrize("maker", [synth.act_decode, synth.act_prefill, synth.act_quant])
def test_matches_independent_torch_cpu(maker, ue):
    M, K = 21, 1024
    xb = maker(M, K)
    q, s = oracle.quant_act(xb, oracle.BF16, 128, ue)
    tq, ts = torch_quant_act(synth.bf16_bits_to_f32(xb), ue)
    np.testing.assert_array_equal(q, tq)
    got = unpack_ue8m0(s, K // 128) if ue else s.astype(np.float64)
    np.testing.assert_array_equal(got[:, :M].T, ts.astype(np.float64))


# ------------------------------------------------------------ weight quant --

def test_weight_quant_blocks_and_tail():
    N, K = 200, 384  # partial last row block (rows 128..199), 3 column blocks
    w = synth.weight_f32(N, K)
    w[3, 200] = 0.5  # dominates block (0, 1)
    q, s = oracle.quant_weight(w, oracle.FP32, 128, 128, False)
    assert s.shape == (2, 3)
    for nb in range(2):
        for kb in range(3):
            blk = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            assert s[nb, kb] == np.float32(np.abs(blk).max()) / np.float32(448.0)
    assert q[3, 200] == 0x7E
    # rows of the partial block dequantise to within half a grid step
    deq = decode_codes(q[128:, :]) * np.repeat(s[1], 128)[None, :]
    np.testing.assert_allclose(deq, w[128:, :], atol=float(s[1].max()) * 16)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_weight_quant_matches_torch(dt):
    N, K = 256, 256
    wf = synth.weight_f32(N, K)
    if dt == "bf16":
        wb = synth.f32_to_bf16_bits(wf)
        q, s = oracle.quant_weight(wb, oracle.BF16, 128, 128, True)
        wf = synth.bf16_bits_to_f32(wb)
    else:
        q, s = oracle.quant_weight(wf, oracle.FP32, 128, 128, True)
    t = torch.from_numpy(wf).view(2, 128, 2, 128)
    amax = t.abs().amax(dim=(1, 3))
    ts = torch.exp2(torch.ceil(torch.log2((torch.clamp(amax, min=1e-10) / 448.0).double()))).float()
    y = torch.clamp(t / ts[:, None, :, None], -448, 448)
    tq = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(N, K).numpy()
    np.testing.assert_array_equal(s, ts.numpy())
    np.testing.assert_array_equal(q, tq)
