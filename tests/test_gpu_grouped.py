"""GPU parity of the grouped (MoE) GEMM, masked layout, against the fp64
oracle: every kernel shape (promotion and block-scaled, both orientations,
split-K), ragged / empty / over-full experts, rows past a count left
untouched, and the full-size MoE decode workload on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_group_gb300 import synth
from parity import TORCH_OUT, check_gemm, scales_to_dev, to_dev, to_dev_bits

pytestmark = pytest.mark.gpu

SENTINEL = -32768.0  # exactly representable in bf16, fp16 and fp32


@pytest.fixture(scope="module")
def fp8bq():
    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq as m
    return m


def grouped_problem(E, M_max, N, K, ue):
    xb = synth.moe_act(E, M_max, K)
    qa, sa = oracle.quant_act(xb, oracle.BF16, 128, ue)
    wb = synth.moe_weight_bf16(E, N, K)
    qs = [oracle.quant_weight(wb[e], oracle.BF16, 128, 128, ue) for e in range(E)]
    qw = np.stack([q for q, _ in qs])
    sw = np.stack([s for _, s in qs])
    return qa, sa, qw, sw


def run(fp8bq, qa, sa, qw, sw, counts, ue, out, variant=None):
    E = len(counts)
    o = torch.full((qa.shape[0], qw.shape[1]), SENTINEL, dtype=TORCH_OUT[out], device="cuda")
    fp8bq.fp8bq_grouped_gemm(to_dev(qa), scales_to_dev(sa), to_dev(qw), to_dev(sw),
                             torch.tensor(np.asarray(counts, dtype=np.int32), device="cuda"),
                             fmt="ue8m0" if ue else "fp32", out_dtype=TORCH_OUT[out], out=o,
                             variant=variant)
    torch.cuda.synchronize()
    assert fp8bq.fp8bq_device_status() == 0
    assert E * (qa.shape[0] // E) == qa.shape[0]
    return o.float().cpu().numpy()


def check_grouped(got, ref, counts, M_max, out, what):
    for e, c in enumerate(counts):
        c = min(max(int(c), 0), M_max)
        r0 = e * M_max
        if c:
            check_gemm(got[r0:r0 + c], ref[r0:r0 + c], out, f"{what} expert {e}")
        assert np.all(got[r0 + c:r0 + M_max] == SENTINEL), f"{what}: expert {e} wrote past its count"


VARIANTS = ([("swap", bn, s, 0) for bn in (16, 32, 64, 128) for s in (1, 2)] +
            [("swap64", bn, s, 0) for bn in (16, 32) for s in (1, 2)] +
            [("normal", bn, s, 0) for bn in (128, 256) for s in (1, 3)] +
            [("swap", bn, s, 1) for bn in (16, 32, 64, 128) for s in (1, 2)] +
            [("normal", bn, s, 1) for bn in (128, 256) for s in (1, 2)])


@pytest.mark.parametrize("kind,bn,split,mx", VARIANTS)
@pytest.mark.parametrize("ue", [False, True])
def test_grouped_variants(fp8bq, kind, bn, split, mx, ue):
    if mx and not ue:
        pytest.skip("the block-scaled MMA takes UE8M0 scales")
    # five experts: ragged, empty, full, over-full (clamped), one row
    E, M_max, N, K = 5, 136, 256, 1024
    counts = [77, 0, 136, 500, 1]
    qa, sa, qw, sw = grouped_problem(E, M_max, N, K, ue)
    ref = oracle.grouped_gemm(qa, sa, qw, sw, counts, ue)
    v = fp8bq.make_variant(kind, bn, split, 0, mx)
    for out in ("bf16", "fp32"):
        got = run(fp8bq, qa, sa, qw, sw, counts, ue, out, v)
        check_grouped(got, ref, counts, M_max, out, f"{kind}/{bn}/{split}/mx{mx} {out}")


@pytest.mark.parametrize("E,M_max,N,K,ue", [(1, 8, 128, 128, False), (3, 4, 384, 512, True),
                                            (8, 24, 512, 2048, True), (2, 260, 768, 512, False)])
def test_grouped_default_variant(fp8bq, E, M_max, N, K, ue):
    rng = np.random.default_rng(E * 1000 + M_max)
    counts = rng.integers(0, M_max + 1, size=E)
    counts[0] = M_max
    qa, sa, qw, sw = grouped_problem(E, M_max, N, K, ue)
    ref = oracle.grouped_gemm(qa, sa, qw, sw, counts, ue)
    for out in ("bf16", "fp16"):
        got = run(fp8bq, qa, sa, qw, sw, counts, ue, out)
        check_grouped(got, ref, counts, M_max, out, f"default {E}x{M_max}x{N}x{K} {out}")


def test_grouped_all_empty_and_errors(fp8bq):
    E, M_max, N, K = 4, 8, 128, 256
    qa, sa, qw, sw = grouped_problem(E, M_max, N, K, True)
    got = run(fp8bq, qa, sa, qw, sw, [0, 0, 0, 0], True, "bf16")
    assert np.all(got == SENTINEL)
    d = (to_dev(qa), scales_to_dev(sa), to_dev(qw), to_dev(sw))
    cnt = torch.zeros(E, dtype=torch.int32, device="cuda")
    # stream-K is not offered for grouped problems
    with pytest.raises(fp8bq.Fp8bqError):
        fp8bq.fp8bq_grouped_gemm(*d, cnt, fmt="ue8m0", variant=fp8bq.make_variant("swap", 16, 0))
    # rows per expert must be a multiple of 4
    with pytest.raises(fp8bq.Fp8bqError):
        fp8bq.fp8bq_grouped_gemm(d[0][:E * 6], d[1], d[2], d[3], cnt, fmt="ue8m0")
    # a null counts pointer is rejected before any launch
    st = fp8bq.lib().fp8bq_grouped_gemm(E, M_max, N, K, None, d[0].data_ptr(), d[1].data_ptr(),
                                        d[2].data_ptr(), d[3].data_ptr(), 128, 128, 128, 1, 0,
                                        d[0].data_ptr(), None, 0, None)
    assert st != 0


@pytest.mark.parametrize("N,K", synth.MOE_NK)
def test_grouped_moe_decode_full_size_sampled(fp8bq, N, K):
    """The MoE decode workload at full size (32 local experts, 128 tokens
    routed top-8 of 256): the first and last valid row of every expert, all
    N columns, plus the untouched rows past each count."""
    E = synth.MOE_E_LOCAL
    counts = synth.moe_counts(E, synth.MOE_TOKENS[0])
    M_max = int((counts.max() + 3) // 4 * 4)
    xb = synth.moe_act(E, M_max, K)
    wb = synth.moe_weight_bf16(E, N, K)
    x = to_dev_bits(xb)
    aq, as_ = fp8bq.fp8bq_quant_act(x, "ue8m0")
    wq = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    ws = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device="cuda")
    for e in range(E):
        fp8bq.fp8bq_quant_weight(to_dev_bits(wb[e]), "ue8m0", q=wq[e], s=ws[e])
    o = torch.full((E * M_max, N), SENTINEL, dtype=torch.bfloat16, device="cuda")
    fp8bq.fp8bq_grouped_gemm(aq, as_, wq, ws, torch.from_numpy(counts).cuda(), fmt="ue8m0",
                             out_dtype=torch.bfloat16, out=o)
    torch.cuda.synchronize()
    got = o.float().cpu().numpy()
    qa, sa = oracle.quant_act(xb, oracle.BF16, 128, True)
    for e in range(E):
        c = int(counts[e])
        r0 = e * M_max
        assert np.all(got[r0 + c:r0 + M_max] == SENTINEL)
        if c == 0:
            continue
        qw, sw = oracle.quant_weight(wb[e], oracle.BF16, 128, 128, True)
        for r in sorted({r0, r0 + c - 1}):
            ref = oracle.gemm(qa, sa, qw, sw, True, rows=(r, 1))
            check_gemm(got[r:r + 1], ref, "bf16", f"moe {N}x{K} expert {e} row {r - r0}")


@pytest.mark.parametrize("E,M_max,N,K,xdt", [(5, 136, 256, 1024, "bf16"), (4, 24, 384, 512, "fp16"),
                                             (3, 260, 768, 2048, "bf16")])
def test_grouped_linear(fp8bq, E, M_max, N, K, xdt):
    """Quant of the occupied rows + grouped GEMM in one call.  The rows past
    each count hold NaN: they must be neither read nor stored."""
    rng = np.random.default_rng(E + M_max)
    counts = rng.integers(0, M_max + 1, size=E).astype(np.int32)
    counts[0] = M_max
    if E > 2:
        counts[1] = 0
    xb = synth.moe_act(E, M_max, K)
    if xdt == "fp16":
        xb = synth.f32_to_f16_bits((xb.astype(np.uint32) << 16).view(np.float32))
    nan_bits = 0x7FC0 if xdt == "bf16" else 0x7E00
    for e in range(E):
        xb[e * M_max + counts[e]:(e + 1) * M_max] = nan_bits
    wb = synth.moe_weight_bf16(E, N, K)
    tdt = torch.bfloat16 if xdt == "bf16" else torch.float16
    wq = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    ws = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device="cuda")
    for e in range(E):
        fp8bq.fp8bq_quant_weight(to_dev_bits(wb[e]), "ue8m0", q=wq[e], s=ws[e])
    o = torch.full((E * M_max, N), SENTINEL, dtype=torch.bfloat16, device="cuda")
    fp8bq.fp8bq_grouped_linear(to_dev_bits(xb, tdt), wq, ws, torch.from_numpy(counts).cuda(),
                               fmt="ue8m0", out_dtype=torch.bfloat16, out=o)
    torch.cuda.synchronize()
    assert fp8bq.fp8bq_device_status() == 0
    got = o.float().cpu().numpy()
    # the oracle quantises the occupied rows (padding rows set to 0 so that its
    # finite-input precondition holds; they are not used)
    xo = xb.copy()
    for e in range(E):
        xo[e * M_max + counts[e]:(e + 1) * M_max] = 0
    qa, sa = oracle.quant_act(xo, oracle.BF16 if xdt == "bf16" else oracle.FP16, 128, True)
    qs = [oracle.quant_weight(wb[e], oracle.BF16, 128, 128, True) for e in range(E)]
    ref = oracle.grouped_gemm(qa, sa, np.stack([q for q, _ in qs]), np.stack([s for _, s in qs]),
                              counts, True)
    check_grouped(got, ref, counts, M_max, "bf16", f"grouped linear {E}x{M_max}x{N}x{K} {xdt}")
