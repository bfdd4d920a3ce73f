"""GPU parity of activation and weight quantisation against the oracle:
codes and scales bit-exact, padding included."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_group_gb300 import synth
from parity import scales_bits, to_dev, to_dev_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8bq():
    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq as m
    return m


def run_act(fp8bq, xb, fp16, ue):
    x = to_dev_bits(xb, torch.float16 if fp16 else torch.bfloat16)
    q, s = fp8bq.fp8bq_quant_act(x, "ue8m0" if ue else "fp32")
    torch.cuda.synchronize()
    return q.cpu().numpy(), scales_bits(s)


@pytest.mark.parametrize("ue", [False, True])
@pytest.mark.parametrize("fp16", [False, True])
@pytest.mark.parametrize("M,K", [(1, 128), (3, 640), (5, 512), (37, 1536), (130, 7168),
                                 (64, 18432), (9, 1152)])
def test_act_quant_bit_exact(fp8bq, M, K, fp16, ue):
    x = synth.normal((M, K), seed=M * 7 + K)
    synth.group_spikes(x, 128, seed=5, row_period=3, row_phase=1)
    xb = synth.f32_to_f16_bits(x) if fp16 else synth.f32_to_bf16_bits(x)
    q, s = run_act(fp8bq, xb, fp16, ue)
    rq, rs = oracle.quant_act(xb, oracle.FP16 if fp16 else oracle.BF16, 128, ue)
    np.testing.assert_array_equal(q, rq)
    np.testing.assert_array_equal(s, rs.view(np.uint32))


@pytest.mark.parametrize("ue", [False, True])
def test_act_quant_every_bf16_value_through_the_converter(fp8bq, ue):
    """Groups whose amax is 448 have s = 1 in both modes, so their other 127
    elements reach the fp8 conversion unchanged: every finite bf16 value in
    [-448, 448] is checked against the oracle's encoder."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = synth.bf16_bits_to_f32(bits)
    keep = bits[np.isfinite(vals) & (np.abs(vals) <= 448)]
    per = 127
    G = (keep.size + per - 1) // per
    groups = np.zeros((G, 128), dtype=np.uint16)
    flat = np.concatenate([keep, np.zeros(G * per - keep.size, dtype=np.uint16)])
    groups[:, 1:] = flat.reshape(G, per)
    groups[:, 0] = synth.f32_to_bf16_bits(np.array([448.0], dtype=np.float32))[0]
    K = 1024
    rows = (G + 7) // 8
    xb = np.zeros((rows * 8, 128), dtype=np.uint16)
    xb[:G] = groups
    xb[G:, 0] = groups[0, 0]
    xb = xb.reshape(rows, K)
    q, s = run_act(fp8bq, xb, False, ue)
    rq, rs = oracle.quant_act(xb, oracle.BF16, 128, ue)
    np.testing.assert_array_equal(q, rq)
    np.testing.assert_array_equal(s, rs.view(np.uint32))


def oracle_quant_rows(xb, ue, chunk=512, threads=16):
    """The oracle's quantisation of every row, in parallel row chunks (rows are
    independent; chunks are multiples of 4 rows, so each chunk's column-major
    scale block is a column slice of the whole)."""
    M = xb.shape[0]
    starts = list(range(0, M, chunk))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda r0: oracle.quant_act(np.ascontiguousarray(xb[r0:r0 + chunk]),
                                                        oracle.BF16, 128, ue), starts))
    q = np.concatenate([p[0] for p in parts], axis=0)
    s = np.concatenate([p[1].view(np.uint32) for p in parts], axis=1)
    return q, s


@pytest.mark.parametrize("ue", [False, True])
@pytest.mark.parametrize("M", [1, 64, 1024, 4096, 16384])
@pytest.mark.parametrize("K", [1536, 7168, 18432])
def test_act_quant_full_size_every_element(fp8bq, M, K, ue):
    """The standalone-quant workload at full size: every code and scale vs the
    oracle, and the padding rows of the scale buffer zero."""
    xb = synth.act_quant(M, K)
    q, s = run_act(fp8bq, xb, False, ue)
    Mp = (M + 3) // 4 * 4
    G = K // 128
    cols = (G + 3) // 4 if ue else G
    assert s.shape == (cols, Mp)
    assert np.all(s[:, M:] == 0)
    rq, rs = oracle_quant_rows(xb, ue)
    np.testing.assert_array_equal(q, rq)
    np.testing.assert_array_equal(s[:, :M], rs[:, :M])


@pytest.mark.parametrize("ue", [False, True])
@pytest.mark.parametrize("dt", ["f32", "bf16", "fp16"])
@pytest.mark.parametrize("N,K", [(128, 128), (200, 384), (1536, 1536), (320, 640)])
def test_weight_quant_bit_exact(fp8bq, N, K, dt, ue):
    wf = synth.weight_f32(N, K, seed=N + K)
    if dt == "f32":
        host, code, dev = wf, oracle.FP32, to_dev(wf)
    elif dt == "bf16":
        host = synth.f32_to_bf16_bits(wf)
        code, dev = oracle.BF16, to_dev_bits(host, torch.bfloat16)
    else:
        host = synth.f32_to_f16_bits(wf)
        code, dev = oracle.FP16, to_dev_bits(host, torch.float16)
    q, s = fp8bq.fp8bq_quant_weight(dev, "ue8m0" if ue else "fp32")
    torch.cuda.synchronize()
    rq, rs = oracle.quant_weight(host, code, 128, 128, ue)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_quant_weight_decode_shapes(fp8bq):
    """The decode-sweep weight shapes at full size, sampled blocks."""
    for N, K in synth.DECODE_NK:
        wb = synth.weight_bf16(N, K)
        q, s = fp8bq.fp8bq_quant_weight(to_dev_bits(wb, torch.bfloat16), "ue8m0")
        torch.cuda.synchronize()
        q = q.cpu().numpy()
        s = s.cpu().numpy()
        rng = np.random.default_rng(N)
        for nb, kb in [(0, 0), (N // 128 - 1, K // 128 - 1)] + [
                (int(a), int(b)) for a, b in zip(rng.integers(0, N // 128, 4),
                                                 rng.integers(0, K // 128, 4))]:
            blk = np.ascontiguousarray(wb[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128])
            rq, rs = oracle.quant_weight(blk, oracle.BF16, 128, 128, True)
            np.testing.assert_array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128], rq)
            assert s[nb, kb] == rs[0, 0]


def test_bounded_wait_times_out_and_reports(fp8bq):
    assert fp8bq.fp8bq_device_status() == 0
    fp8bq.fp8bq_selftest_wait_timeout(20_000_000)  # 20 ms, nothing ever arrives
    assert fp8bq.fp8bq_device_status() == 7        # FP8BQ_ERR_DEVICE_TIMEOUT
    assert fp8bq.fp8bq_device_status() == 0        # read clears it
    # the context is still usable
    x = to_dev_bits(synth.act_small(4, 256))
    fp8bq.fp8bq_quant_act(x, "fp32")
    torch.cuda.synchronize()


def test_fp32_converter_every_pattern(fp8bq):
    """Every fp32 bit pattern in [-448, 448] (both signs, zeros and
    subnormals included) through the GPU's e4m3 conversion.  In fp32 weight
    blocks whose first element is 448 the scale is 448/448 = 1 exactly, so
    each of the other 16383 elements reaches the conversion unchanged; its
    code must be the oracle's encoding of the same value."""
    per = 128 * 128 - 1
    top = 0x43E00000  # 448.0
    n_pos = top + 1   # patterns 0 .. 448.0 of one sign
    blocks = 2048
    chunk = blocks * per
    dev_w = torch.empty((blocks * 128, 128), dtype=torch.float32, device="cuda")
    dev_q = torch.empty((blocks * 128, 128), dtype=torch.uint8, device="cuda")
    dev_s = torch.empty((blocks, 1), dtype=torch.float32, device="cuda")
    host = np.empty((blocks, 128 * 128), dtype=np.uint32)
    host[:, 0] = top
    checked = 0

    def oracle_codes(w, nb):
        bounds = np.linspace(0, nb, 17).astype(int) * 128
        with ThreadPoolExecutor(max_workers=16) as ex:
            parts = list(ex.map(lambda r: oracle.quant_weight(w[r[0]:r[1]], oracle.FP32)[0],
                                [(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]))
        return np.concatenate(parts, axis=0)

    for sign in (0, 0x80000000):
        for start in range(0, n_pos, chunk):
            cnt = min(chunk, n_pos - start)
            nb = (cnt + per - 1) // per
            body = np.full(nb * per, top, dtype=np.uint32)  # padding repeats 448
            body[:cnt] = np.arange(start, start + cnt, dtype=np.uint32) | np.uint32(sign)
            host[:nb, 1:] = body.reshape(nb, per)
            w = host[:nb].view(np.float32).reshape(nb * 128, 128)
            dev_w[:nb * 128].copy_(torch.from_numpy(w))
            fp8bq.fp8bq_quant_weight(dev_w[:nb * 128], "fp32", q=dev_q[:nb * 128], s=dev_s[:nb])
            q = dev_q[:nb * 128].cpu().numpy()
            s = dev_s[:nb].cpu().numpy()
            assert np.all(s == 1.0)
            rq = oracle_codes(w, nb)
            if not np.array_equal(q, rq):
                bad = np.flatnonzero(q.reshape(-1) != rq.reshape(-1))[:5]
                vals = w.reshape(-1)[bad]
                raise AssertionError(f"codes differ at {vals!r}: gpu {q.reshape(-1)[bad]}, "
                                     f"oracle {rq.reshape(-1)[bad]}")
            checked += cnt
    assert checked == 2 * n_pos


@pytest.mark.parametrize("ue", [False, True])
@pytest.mark.parametrize("amax", [1.0, 3.0, 0.3, 1000.0, 7.0e-3, 250.0, 1.0e-6])
def test_act_quant_every_bf16_value_per_scale(fp8bq, amax, ue):
    """Groups whose first element is A (a bf16 value) have s = fp32(A/448)
    (UE8M0: the next power of two), which is not a power of two in fp32 mode,
    so each of the other 127 elements goes through the IEEE division x/s and
    the e4m3 conversion: every finite bf16 value with |x| <= A is checked
    against the oracle for each A."""
    a_bits = synth.f32_to_bf16_bits(np.array([amax], dtype=np.float32))[0]
    a_val = synth.bf16_bits_to_f32(np.array([a_bits], dtype=np.uint16))[0]
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = synth.bf16_bits_to_f32(bits)
    keep = bits[np.isfinite(vals) & (np.abs(vals) <= a_val)]
    per = 127
    G = (keep.size + per - 1) // per
    groups = np.zeros((G, 128), dtype=np.uint16)
    flat = np.concatenate([keep, np.zeros(G * per - keep.size, dtype=np.uint16)])
    groups[:, 1:] = flat.reshape(G, per)
    groups[:, 0] = a_bits
    rows = (G + 7) // 8
    xb = np.zeros((rows * 8, 128), dtype=np.uint16)
    xb[:G] = groups
    xb[G:, 0] = a_bits
    xb = xb.reshape(rows, 1024)
    q, s = run_act(fp8bq, xb, False, ue)
    rq, rs = oracle.quant_act(xb, oracle.BF16, 128, ue)
    np.testing.assert_array_equal(q, rq)
    np.testing.assert_array_equal(s, rs.view(np.uint32))


def _near_midpoint_pairs(n_scales=2000, seed=21, ulps=8):
    """(A, x) bf16 pairs whose quotient fp32(x / fp32(A/448)) lies within
    `ulps` fp32 ulps of an e4m3 rounding boundary (the midpoint of two
    adjacent normal e4m3 values: the 20 mantissa bits e4m3 drops equal
    0x80000), found by scanning every positive bf16 x <= A for seeded A."""
    rng = np.random.default_rng(seed)
    bits = np.arange(0x0080, 0x7F80, dtype=np.uint32).astype(np.uint16)  # positive normals
    vals = synth.bf16_bits_to_f32(bits)
    a_bits = rng.choice(bits[(vals >= 1e-3) & (vals <= 1e4)], size=n_scales, replace=False)
    pairs = []
    for ab in a_bits:
        a = synth.bf16_bits_to_f32(np.array([ab], dtype=np.uint16))[0]
        s = np.float32(a) / np.float32(448.0)  # IEEE fp32 division
        xs = bits[vals <= a]
        q = synth.bf16_bits_to_f32(xs) / s
        u = q.view(np.uint32)
        d = np.abs((u & np.uint32(0xFFFFF)).astype(np.int64) - 0x80000)
        hit = (d <= ulps) & (q >= np.float32(2.0 ** -6))
        pairs += [(int(ab), int(x)) for x in xs[hit]]
    return pairs


def test_act_quant_fp32_scale_near_rounding_boundaries(fp8bq):
    """fp32 scales: inputs whose quotient x/s falls within a few fp32 ulps of
    an e4m3 rounding boundary (including exact ties) -- where a product by
    the reciprocal would round to another code than the IEEE quotient -- each
    in a group whose amax A sets s, with both signs; codes and scales
    bit-exact against the oracle."""
    pairs = _near_midpoint_pairs()
    assert len(pairs) > 500
    by_a = {}
    for ab, x in pairs:
        by_a.setdefault(ab, []).append(x)
    groups = []
    for ab, xs in by_a.items():
        for i in range(0, len(xs), 63):
            g = np.zeros(128, dtype=np.uint16)
            g[0] = ab
            chunk = np.array(xs[i:i + 63], dtype=np.uint16)
            g[1:1 + chunk.size] = chunk
            g[64:64 + chunk.size] = chunk | np.uint16(0x8000)  # negatives
            groups.append(g)
    rows = (len(groups) + 7) // 8
    xb = np.zeros((rows * 8, 128), dtype=np.uint16)
    xb[:len(groups)] = np.stack(groups)
    xb = xb.reshape(rows, 1024)
    q, s = run_act(fp8bq, xb, False, False)
    rq, rs = oracle.quant_act(xb, oracle.BF16, 128, False)
    np.testing.assert_array_equal(q, rq)
    np.testing.assert_array_equal(s, rs.view(np.uint32))
