"""GPU parity of the block-scaled GEMM (every variant) and the fused linear
layer against the fp64 oracle, within the stated element-wise / Frobenius
bounds.  Inputs are quantised by the oracle on the host, so the GEMM is
checked independently of the GPU quant kernel."""
import functools

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_group_gb300 import synth
from parity import (TORCH_OUT, check_gemm, oracle_full, oracle_rows, quantised_problem,
                    sample_rows, scales_to_dev, to_dev, to_dev_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8bq():
    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq as m
    return m


def upload(qa, sa, qw, sw):
    return to_dev(qa), scales_to_dev(sa), to_dev(qw), to_dev(sw)


# split 0 = stream-K (equal shares of the (tile, K slab) units per CTA)
# swap64: 64 weight rows per tile (MMA M = 64)
VARIANTS = ([("swap", bn, s) for bn in (16, 32, 64, 128) for s in (0, 1, 2, 3)] +
            [("swap64", bn, s) for bn in (16, 32) for s in (0, 1, 2, 3)] +
            [("normal", bn, s) for bn in (128, 256) for s in (0, 1, 2, 5)])


@pytest.mark.parametrize("kind,bn,split", VARIANTS)
@pytest.mark.parametrize("M,N,K,ue", [(1, 128, 128, False), (5, 320, 640, True),
                                      (77, 256, 1024, False), (130, 384, 768, True)])
def test_variants_small(fp8bq, kind, bn, split, M, N, K, ue):
    if split > K // 128:
        pytest.skip("more splits than K slabs")
    xb, qa, sa, qw, sw = quantised_problem(M, N, K, ue, synth.act_decode)
    ref = oracle_full(qa, sa, qw, sw, ue)
    d = upload(qa, sa, qw, sw)
    v = fp8bq.make_variant(kind, bn, split)
    for out in ("bf16", "fp32"):
        o = fp8bq.fp8bq_gemm_variant(*d, v, fmt="ue8m0" if ue else "fp32",
                                     out_dtype=TORCH_OUT[out])
        torch.cuda.synchronize()
        check_gemm(o.float().cpu().numpy(), ref, out, f"{kind}/{bn}/{split} {M}x{N}x{K} {out}")


# block-scaled MMA: the tensor core applies the UE8M0 scales (K % 512 == 0)
MX_VARIANTS = ([("swap", bn, s) for bn in (16, 32, 64, 128) for s in (0, 1, 2, 3)] +
               [("normal", bn, s) for bn in (128, 256) for s in (0, 1, 2, 3)])


@pytest.mark.parametrize("kind,bn,split", MX_VARIANTS)
@pytest.mark.parametrize("M,N,K", [(1, 128, 512), (5, 320, 1024), (77, 256, 2048),
                                   (130, 384, 1536), (300, 640, 1024)])
def test_mx_variants_small(fp8bq, kind, bn, split, M, N, K):
    xb, qa, sa, qw, sw = quantised_problem(M, N, K, True, synth.act_decode)
    ref = oracle_full(qa, sa, qw, sw, True)
    d = upload(qa, sa, qw, sw)
    v = fp8bq.make_variant(kind, bn, split, 0, 1)
    for out in ("bf16", "fp32"):
        o = fp8bq.fp8bq_gemm_variant(*d, v, fmt="ue8m0", out_dtype=TORCH_OUT[out])
        torch.cuda.synchronize()
        check_gemm(o.float().cpu().numpy(), ref, out, f"mx {kind}/{bn}/{split} {M}x{N}x{K} {out}")


@pytest.mark.parametrize("split,grid", [(7, 0), (0, 0), (0, 13), (1, 5)])
def test_mx_bit_stable_and_persistent(fp8bq, split, grid):
    M, N, K = 24, 1024, 4096
    xb, qa, sa, qw, sw = quantised_problem(M, N, K, True, synth.act_full_grid)
    d = upload(qa, sa, qw, sw)
    v = fp8bq.make_variant("swap", 32, split, grid, 1)
    outs = [fp8bq.fp8bq_gemm_variant(*d, v, fmt="ue8m0", out_dtype=torch.float32)
            for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    check_gemm(outs[0].cpu().numpy(), oracle_full(qa, sa, qw, sw, True), "fp32",
               f"mx split {split} grid {grid}")


def test_mx_rejections(fp8bq):
    for (K, ue, kind) in ((512, False, "swap"),    # fp32 scales
                          (640, True, "swap"),     # K not a multiple of 512
                          (512, True, "swap64")):  # M = 128 MMAs only
        xb, qa, sa, qw, sw = quantised_problem(16, 256, K, ue, synth.act_decode)
        d = upload(qa, sa, qw, sw)
        with pytest.raises(fp8bq.Fp8bqError) as e:
            fp8bq.fp8bq_gemm_variant(*d, fp8bq.make_variant(kind, 16, 1, 0, 1),
                                     fmt="ue8m0" if ue else "fp32", out_dtype=torch.float32)
        assert e.value.status == 4


@pytest.mark.parametrize("grid", [1, 3, 7])
def test_persistent_grid_loops_over_items(fp8bq, grid):
    M, N, K = 40, 640, 1280
    xb, qa, sa, qw, sw = quantised_problem(M, N, K, True, synth.act_prefill)
    ref = oracle_full(qa, sa, qw, sw, True)
    d = upload(qa, sa, qw, sw)
    for v in (fp8bq.make_variant("swap", 64, 3, grid), fp8bq.make_variant("normal", 128, 2, grid),
              fp8bq.make_variant("swap", 32, 0, grid), fp8bq.make_variant("normal", 256, 0, grid)):
        o = fp8bq.fp8bq_gemm_variant(*d, v, fmt="ue8m0", out_dtype=torch.float32)
        torch.cuda.synchronize()
        check_gemm(o.cpu().numpy(), ref, "fp32", f"grid {grid} {v.as_dict()}")


@pytest.mark.parametrize("split,grid", [(7, 0), (0, 0), (0, 13)])
def test_split_k_is_bit_stable_and_reusable(fp8bq, split, grid):
    M, N, K = 24, 1024, 2048
    xb, qa, sa, qw, sw = quantised_problem(M, N, K, False, synth.act_decode)
    d = upload(qa, sa, qw, sw)
    v = fp8bq.make_variant("swap", 32, split, grid)
    outs = [fp8bq.fp8bq_gemm_variant(*d, v, out_dtype=torch.float32) for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    check_gemm(outs[0].cpu().numpy(), oracle_full(qa, sa, qw, sw, False), "fp32",
               f"split {split} grid {grid}")


def test_fp16_output(fp8bq):
    M, N, K = 33, 512, 1024
    xb, qa, sa, qw, sw = quantised_problem(M, N, K, True, synth.act_full_grid)
    ref = oracle_full(qa, sa, qw, sw, True)
    o = fp8bq.fp8bq_gemm(*upload(qa, sa, qw, sw), fmt="ue8m0", out_dtype=torch.float16)
    torch.cuda.synchronize()
    check_gemm(o.float().cpu().numpy(), ref, "fp16")


def test_small_config_full(fp8bq):
    """M=16, N=K=1536: bf16 N(0,1) activations with fp32 scales, fp32
    N(0,0.02) weights, bf16 output -- every element."""
    M, N, K = 16, 1536, 1536
    xb, qa, sa, qw, sw = quantised_problem(M, N, K, False, synth.act_small)
    ref = oracle_full(qa, sa, qw, sw, False)
    o = fp8bq.fp8bq_gemm(*upload(qa, sa, qw, sw), fmt="fp32", out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    check_gemm(o.float().cpu().numpy(), ref, "bf16", "small config")
    # the same through the GPU quant kernels and the fused linear entry point
    w = synth.weight_f32(N, K)
    wq, ws = fp8bq.fp8bq_quant_weight(to_dev(w), "fp32")
    o2 = fp8bq.fp8bq_linear(to_dev_bits(xb), wq, ws, fmt="fp32", out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    check_gemm(o2.float().cpu().numpy(), ref, "bf16", "small config linear")


@functools.lru_cache(maxsize=3)
def _decode_weights(N, K):
    """Oracle-quantised decode weights (UE8M0), on the host and the device."""
    wb = synth.weight_bf16(N, K)
    qw, sw = oracle.quant_weight(wb, oracle.BF16, 128, 128, True)
    return qw, sw, to_dev(qw), to_dev(sw)


@pytest.mark.parametrize("N,K", synth.DECODE_NK)
@pytest.mark.parametrize("M", synth.DECODE_M)
def test_decode_every_element(fp8bq, N, K, M):
    """The decode sweep at full size (UE8M0, bf16 out): every output element,
    in the variant the table selects, and with the table's token tile and split
    in both scale paths (CUDA-core promotion, block-scaled MMA) and, for token
    tiles up to 32, with 64-row weight tiles."""
    qw, sw, dqw, dsw = _decode_weights(N, K)
    qa, sa = oracle.quant_act(synth.act_decode(M, K), oracle.BF16, 128, True)
    ref = oracle_full(qa, sa, qw, sw, True)
    da, dsa = to_dev(qa), scales_to_dev(sa)
    o = fp8bq.fp8bq_gemm(da, dsa, dqw, dsw, fmt="ue8m0", out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    check_gemm(o.float().cpu().numpy(), ref, "bf16", f"decode {M}x{N}x{K} (table)")
    sel = fp8bq.fp8bq_select_variant(M, N, K, "ue8m0", "bf16")
    bn, split = sel["block_n"], sel["split"]
    others = [("swap", 0), ("swap", 1)] + ([("swap64", 0)] if bn <= 32 else [])
    for kind, mx in others:
        v = fp8bq.make_variant(kind, bn, split, 0, mx)
        o = fp8bq.fp8bq_gemm_variant(da, dsa, dqw, dsw, v, fmt="ue8m0", out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        check_gemm(o.float().cpu().numpy(), ref, "bf16", f"decode {M}x{N}x{K} {v.as_dict()}")


@pytest.mark.parametrize("N,K", synth.PREFILL_NK)
@pytest.mark.parametrize("M", synth.PREFILL_M)
def test_prefill_full_size_sampled(fp8bq, N, K, M):
    """Prefill sweep at full size (fp32 scales, bf16 and fp32 out): all N
    columns of 64 seeded rows plus the tile-boundary rows, through the GEMM
    on oracle-quantised inputs and through the fused linear entry point (GPU
    quant of the same bf16 input, then the GEMM with its weight prefetch)."""
    xb, qa, sa, qw, sw = quantised_problem(M, N, K, False, synth.act_prefill, weight="bf16")
    d = upload(qa, sa, qw, sw)
    rows = sample_rows(M, 64)
    ref = oracle_rows(qa, sa, qw, sw, False, rows)
    x = to_dev_bits(xb)
    for out in ("bf16", "fp32"):
        o = fp8bq.fp8bq_gemm(*d, fmt="fp32", out_dtype=TORCH_OUT[out])
        lin = fp8bq.fp8bq_linear(x, d[2], d[3], fmt="fp32", out_dtype=TORCH_OUT[out])
        torch.cuda.synchronize()
        check_gemm(o.float().cpu().numpy()[rows], ref, out, f"prefill {M}x{N}x{K} {out}")
        check_gemm(lin.float().cpu().numpy()[rows], ref, out, f"prefill linear {M}x{N}x{K} {out}")


_GRID_W = {}   # (N, K) -> (oracle codes, oracle scales, device codes, device scales)
_GRID_REF = {}  # (N, K) -> {row: fp64 oracle row}


def _grid_weights(fp8bq, N, K):
    if (N, K) not in _GRID_W:
        wb = synth.weight_bf16_blocked(N, K)
        qw, sw = oracle.quant_weight(wb, oracle.BF16, 128, 128, True)
        wq, ws = fp8bq.fp8bq_quant_weight(to_dev_bits(wb), "ue8m0")
        _GRID_W[(N, K)] = (qw, sw, wq, ws)
    return _GRID_W[(N, K)]


@functools.lru_cache(maxsize=3)
def _grid_act(K):
    # rows of the blocked generator depend only on (seed, row): the M-row
    # input of every grid point is the first M rows of this one
    return synth.act_full_grid_blocked(max(synth.M_GRID), K)


def _grid_ref(N, K, qw, sw, rows):
    """Oracle rows of the full-grid problem (N, K), cached across M."""
    cache = _GRID_REF.setdefault((N, K), {})
    need = [r for r in rows if r not in cache]
    if need:
        xb = np.ascontiguousarray(_grid_act(K)[need])
        qa, sa = oracle.quant_act(xb, oracle.BF16, 128, True)
        ref = oracle_full(qa, sa, qw, sw, True)
        for i, r in enumerate(need):
            cache[r] = ref[i]
    return np.stack([cache[r] for r in rows])


@pytest.mark.parametrize("M", synth.M_GRID)
@pytest.mark.parametrize("N,K", synth.FULL_NK)
def test_linear_full_grid(fp8bq, N, K, M):
    """The full grid through the fused linear entry point (UE8M0, fp16 and
    bf16 out), at every M point and (N,K), in the kernels the table selects
    for each; the reference quantises with the oracle on the host.  Every
    element for M <= 128, else all columns of 64 seeded rows plus the
    tile-boundary rows."""
    qw, sw, wq, ws = _grid_weights(fp8bq, N, K)
    xb = _grid_act(K)[:M]
    rows = list(range(M)) if M <= 128 else sample_rows(M, 64)
    ref = _grid_ref(N, K, qw, sw, rows)
    x = to_dev_bits(xb)
    for out in ("fp16", "bf16"):
        o = fp8bq.fp8bq_linear(x, wq, ws, fmt="ue8m0", out_dtype=TORCH_OUT[out])
        torch.cuda.synchronize()
        sel = fp8bq.fp8bq_select_variant(M, N, K, "ue8m0", out)
        check_gemm(o.float().cpu().numpy()[rows], ref, out,
                   f"linear {M}x{N}x{K} {out} {sel}")


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (5, 384, 1024), (16, 1024, 2048),
                                   (24, 640, 1536), (32, 4096, 7168), (16, 18432, 7168)])
@pytest.mark.parametrize("xdt", ["bf16", "fp16"])
def test_linear_fused_quant(fp8bq, M, N, K, xdt, monkeypatch):
    """UE8M0 with a swap-AB tile of 16/32 tokens and FP8BQ_LINEAR_FUSE=1:
    fp8bq_linear runs one block-scaled launch that quantises its own
    activation tiles.  Its output equals (bit for bit) the standalone quant
    followed by the block-scaled GEMM of the same tile and split, and matches
    the oracle; the default (unfused) path matches the oracle too."""
    tdt = torch.bfloat16 if xdt == "bf16" else torch.float16
    xb = synth.act_full_grid(M, K)
    if xdt == "fp16":  # the same values as fp16 bit patterns
        xb = synth.f32_to_f16_bits((xb.astype(np.uint32) << 16).view(np.float32))
    wb = synth.weight_bf16(N, K)
    x = to_dev_bits(xb, tdt)
    wq, ws = fp8bq.fp8bq_quant_weight(to_dev_bits(wb), "ue8m0")
    sel = fp8bq.fp8bq_select_variant(M, N, K, "ue8m0", "bf16")
    if sel["kind"] != "swap" or sel["block_n"] > 32:
        pytest.skip("the table picks a tile the fused path does not cover")
    monkeypatch.setenv("FP8BQ_LINEAR_FUSE", "1")
    fused = fp8bq.fp8bq_linear(x, wq, ws, fmt="ue8m0", out_dtype=torch.bfloat16)
    monkeypatch.delenv("FP8BQ_LINEAR_FUSE")
    aq, as_ = fp8bq.fp8bq_quant_act(x, "ue8m0")
    v = fp8bq.make_variant("swap", sel["block_n"], sel["split"], sel["grid"], 1)
    two = fp8bq.fp8bq_gemm_variant(aq, as_, wq, ws, v, fmt="ue8m0", out_dtype=torch.bfloat16)
    unfused = fp8bq.fp8bq_linear(x, wq, ws, fmt="ue8m0", out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(fused, two), "fused linear differs from quant + block-scaled GEMM"
    qw, sw = oracle.quant_weight(wb, oracle.BF16, 128, 128, True)
    qa, sa = oracle.quant_act(xb, oracle.BF16 if xdt == "bf16" else oracle.FP16, 128, True)
    ref = oracle_full(qa, sa, qw, sw, True)
    check_gemm(fused.float().cpu().numpy(), ref, "bf16", f"fused linear {M}x{N}x{K} {xdt}")
    check_gemm(unfused.float().cpu().numpy(), ref, "bf16", f"unfused linear {M}x{N}x{K} {xdt}")


def test_empty_and_errors(fp8bq):
    a = torch.zeros((0, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2, 0), dtype=torch.float32, device="cuda")
    w = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    ws = torch.ones((1, 2), dtype=torch.float32, device="cuda")
    # M = 0 is a no-op (pointers of empty tensors may be null: use a dummy)
    o = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    st = fp8bq.lib().fp8bq_gemm(0, 128, 256, w.data_ptr(), ws.data_ptr(), w.data_ptr(),
                                ws.data_ptr(), 128, 128, 128, 0, 0, w.data_ptr(), None, 0, None)
    assert st == 0
    with pytest.raises(fp8bq.Fp8bqError):
        fp8bq.fp8bq_gemm_variant(w[:, :256], ws, w, ws, fp8bq.make_variant("swap", 48, 1))
    # a too-small workspace is rejected before launching
    M, N, K = 8, 1024, 1024
    qa = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones((8, 8), dtype=torch.float32, device="cuda")
    wq = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sw = torch.ones((8, 8), dtype=torch.float32, device="cuda")
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8bq.Fp8bqError) as e:
        fp8bq.fp8bq_gemm_variant(qa, sa, wq, sw, fp8bq.make_variant("swap", 16, 4),
                                 workspace=small)
    assert e.value.status == 5
