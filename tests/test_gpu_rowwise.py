"""GPU parity of the per-token x per-channel formats (FP8_Dynamic and
W8A8_INT8 of "用 Helion 为 vLLM 构建高性能可移植线性后端", 范围) against the
oracle:

* fp8bq_quant_rows: codes and scales bit-exact (bf16/fp16/fp32 input, e4m3
  and int8 codes, rows longer than the kernel's register cache, K not a
  multiple of 128, every finite bf16 value through the converter);
* fp8bq_gemm_rowwise: every kernel shape (e4m3: swap-AB and normal tiles,
  split-K, stream-K; int8 on the warp-level MMA: swap-AB tiles; int8 as two
  e4m3 planes on the tcgen05 MMA: swap-AB and normal tiles; each with split-K
  and stream-K) on ragged shapes that span several tiles, all output dtypes,
  the extreme int8 codes, and DeepSeek-V3 shapes at full size on sampled rows;
* fp8bq_linear_rowwise: quant + GEMM in one call.
"""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_group_gb300 import synth
from parity import TORCH_OUT, check_gemm, to_dev, to_dev_bits

pytestmark = pytest.mark.gpu

CODES = {"e4m3": False, "int8": True}


@pytest.fixture(scope="module")
def fp8bq():
    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq as m
    return m


def f32_of_bf16(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def quant_on_gpu(fp8bq, x_np, dtype, code):
    if dtype == "fp32":
        x = to_dev(x_np)
    else:
        x = to_dev_bits(x_np, torch.bfloat16 if dtype == "bf16" else torch.float16)
    q, s = fp8bq.fp8bq_quant_rows(x, code)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def make_input(R, K, dtype, seed=0):
    if dtype == "fp32":
        return synth.weight_f32(R, K, seed=seed)
    xb = synth.act_decode(R, K, seed=seed)
    if dtype == "fp16":
        xb = synth.f32_to_f16_bits(f32_of_bf16(xb))
    return xb


ORACLE_DT = {"bf16": oracle.BF16, "fp16": oracle.FP16, "fp32": oracle.FP32}


# ------------------------------------------------------------------- quant --

@pytest.mark.parametrize("code", ["e4m3", "int8"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R,K", [(1, 16), (3, 1040), (64, 7168), (37, 18432), (5, 24576)])
def test_quant_rows_bit_exact(fp8bq, code, dtype, R, K):
    x = make_input(R, K, dtype, seed=R + K)
    q, s = quant_on_gpu(fp8bq, x, dtype, code)
    qo, so = oracle.quant_rows(x, ORACLE_DT[dtype], int8=CODES[code])
    assert np.array_equal(q.view(np.uint8), qo.view(np.uint8)), "codes"
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32)), "scales"


@pytest.mark.parametrize("code", ["e4m3", "int8"])
def test_quant_rows_every_bf16_value(fp8bq, code):
    """All finite bf16 values (shuffled into rows of 256), each row with its
    own amax: codes and scales bit-exact."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    vals = bits[finite]
    vals = np.random.default_rng(7).permutation(vals)
    R = len(vals) // 256
    x = np.ascontiguousarray(vals[:R * 256].reshape(R, 256))
    q, s = quant_on_gpu(fp8bq, x, "bf16", code)
    qo, so = oracle.quant_rows(x, oracle.BF16, int8=CODES[code])
    assert np.array_equal(q.view(np.uint8), qo.view(np.uint8))
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))


def test_quant_rows_weight_workload(fp8bq):
    """Per-channel quant of a DeepSeek-V3 weight (N=4096, K=7168), both codes."""
    w = synth.weight_bf16(4096, 7168)
    for code in ("e4m3", "int8"):
        q, s = quant_on_gpu(fp8bq, w, "bf16", code)
        qo, so = oracle.quant_rows(w, oracle.BF16, int8=CODES[code])
        assert np.array_equal(q.view(np.uint8), qo.view(np.uint8)), code
        assert np.array_equal(s.view(np.uint32), so.view(np.uint32)), code


# -------------------------------------------------------------------- GEMM --

def rowwise_problem(M, N, K, code, seed=0, act=synth.act_decode):
    xb = act(M, K, seed=seed)
    qa, sa = oracle.quant_rows(xb, oracle.BF16, int8=CODES[code])
    qw, sw = oracle.quant_rows(synth.weight_f32(N, K, seed=seed + 1), oracle.FP32,
                               int8=CODES[code])
    return xb, qa, sa, qw, sw


def run_gemm(fp8bq, qa, sa, qw, sw, code, out, variant=None):
    o = fp8bq.fp8bq_gemm_rowwise(to_dev(qa), to_dev(sa), to_dev(qw), to_dev(sw), code,
                                 TORCH_OUT[out], variant=variant)
    torch.cuda.synchronize()
    assert fp8bq.fp8bq_device_status() == 0
    return o.float().cpu().numpy()


E4M3_VARIANTS = ([("swap", bn, s) for bn in (16, 32, 64, 128) for s in (1, 2, 0)] +
                 [("normal", bn, s) for bn in (128, 256) for s in (1, 3, 0)])
INT8_VARIANTS = ([("swap", bn, s, 0) for bn in (8, 16, 32, 64, 128) for s in (1, 3, 0)] +
                 [("swap", bn, s, 1) for bn in (16, 32, 64, 128) for s in (1, 3, 0)] +
                 [("normal", bn, s, 1) for bn in (128, 256) for s in (1, 3, 0)])


@pytest.mark.parametrize("kind,bn,split", E4M3_VARIANTS)
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_gemm_rowwise_e4m3_variants(fp8bq, kind, bn, split, out):
    # ragged everywhere: tokens past whole tiles, weight rows past 128-row
    # tiles (N = 400), a partial last K slab (K = 1040)
    M = 37 if kind == "swap" else 300
    N, K = 400, 1040
    _, qa, sa, qw, sw = rowwise_problem(M, N, K, "e4m3", seed=bn + split)
    got = run_gemm(fp8bq, qa, sa, qw, sw, "e4m3", out, fp8bq.make_variant(kind, bn, split))
    ref = oracle.gemm_rowcol(qa, sa, qw, sw, False)
    check_gemm(got, ref, out, f"e4m3 {kind}/{bn}/s{split}")


@pytest.mark.parametrize("kind,bn,split,planes", INT8_VARIANTS)
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_gemm_rowwise_int8_variants(fp8bq, kind, bn, split, planes, out):
    """planes=0: the warp-level int8 MMA; planes=1: the codes as two e4m3
    planes (16 h, l of q = 16 h + l) on the tcgen05 FP8 MMA."""
    M, N, K = 150, 400, 1040
    _, qa, sa, qw, sw = rowwise_problem(M, N, K, "int8", seed=bn + split,
                                        act=synth.act_prefill)
    got = run_gemm(fp8bq, qa, sa, qw, sw, "int8", out,
                   fp8bq.make_variant(kind, bn, split, 0, planes))
    ref = oracle.gemm_rowcol(qa, sa, qw, sw, True)
    check_gemm(got, ref, out, f"int8 {kind}/{bn}/s{split}/planes={planes}")


def test_gemm_rowwise_int8_extreme_codes(fp8bq):
    """Codes at the ends of the range (-128 is not produced by the quant but
    is a valid int8 input) and every code value, on both int8 kernels: the
    plane split must reproduce q exactly."""
    M, N, K = 64, 256, 512
    rng = np.random.default_rng(5)
    qa = rng.integers(-128, 128, size=(M, K), dtype=np.int16).astype(np.int8)
    qw = rng.integers(-128, 128, size=(N, K), dtype=np.int16).astype(np.int8)
    qa[0, :] = -128
    qw[0, :] = -128
    qa[1, :256] = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    qw[1, :256] = np.arange(127, -129, -1, dtype=np.int16).astype(np.int8)
    sa = np.full(M, 0.01, dtype=np.float32)
    sw = np.full(N, 0.02, dtype=np.float32)
    ref = oracle.gemm_rowcol(qa, sa, qw, sw, True)
    for planes in (0, 1):
        got = run_gemm(fp8bq, qa, sa, qw, sw, "int8", "fp32",
                       fp8bq.make_variant("swap", 64, 1, 0, planes))
        check_gemm(got, ref, "fp32", f"int8 extreme codes planes={planes}")
        # row 0 x column 0: 512 products of (-128)(-128), the largest sum
        assert abs(got[0, 0] - ref[0, 0]) <= 1e-6 * abs(ref[0, 0])


@pytest.mark.parametrize("code", ["e4m3", "int8"])
@pytest.mark.parametrize("out", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("M,N,K", [(1, 16, 16), (1, 7168, 2048), (16, 1536, 1536),
                                   (200, 2048, 7168)])
def test_gemm_rowwise_default_variant(fp8bq, code, out, M, N, K):
    _, qa, sa, qw, sw = rowwise_problem(M, N, K, code, seed=M)
    got = run_gemm(fp8bq, qa, sa, qw, sw, code, out)
    ref = oracle.gemm_rowcol(qa, sa, qw, sw, CODES[code])
    check_gemm(got, ref, out, f"{code} {M}x{N}x{K}")


@pytest.mark.parametrize("code", ["e4m3", "int8"])
@pytest.mark.parametrize("M,N,K", [(8, 18432, 7168), (128, 7168, 18432), (2048, 4096, 7168)])
def test_gemm_rowwise_full_size_sampled(fp8bq, code, M, N, K):
    """DeepSeek-V3 shapes at full size, default kernel shape; all N columns
    of sampled rows (first, last, and rows of the last partial tile)."""
    _, qa, sa, qw, sw = rowwise_problem(M, N, K, code, seed=3, act=synth.act_prefill)
    got = run_gemm(fp8bq, qa, sa, qw, sw, code, "bf16")
    rows = sorted({0, 1, M // 2, M - 2, M - 1} & set(range(M)))
    for r in rows:
        ref = oracle.gemm_rowcol(qa, sa, qw, sw, CODES[code], rows=(r, 1))
        check_gemm(got[r:r + 1], ref, "bf16", f"{code} {M}x{N}x{K} row {r}")


@pytest.mark.parametrize("code", ["e4m3", "int8"])
@pytest.mark.parametrize("xdt", ["bf16", "fp16"])
@pytest.mark.parametrize("M,N,K", [(5, 1536, 1536), (96, 4096, 7168), (300, 1024, 1040)])
def test_linear_rowwise(fp8bq, code, xdt, M, N, K):
    xb = synth.act_decode(M, K, seed=11)
    if xdt == "fp16":
        xb = synth.f32_to_f16_bits(f32_of_bf16(xb))
    w = synth.weight_bf16(N, K)
    qw, sw = fp8bq.fp8bq_quant_rows(to_dev_bits(w), code)
    x = to_dev_bits(xb, torch.bfloat16 if xdt == "bf16" else torch.float16)
    o = fp8bq.fp8bq_linear_rowwise(x, qw, sw, code, torch.bfloat16)
    torch.cuda.synchronize()
    assert fp8bq.fp8bq_device_status() == 0
    qa, sa = oracle.quant_rows(xb, ORACLE_DT[xdt], int8=CODES[code])
    qwo, swo = oracle.quant_rows(w, oracle.BF16, int8=CODES[code])
    assert np.array_equal(qw.cpu().numpy().view(np.uint8), qwo.view(np.uint8))
    ref = oracle.gemm_rowcol(qa, sa, qwo, swo, CODES[code])
    check_gemm(o.float().cpu().numpy(), ref, "bf16", f"linear {code} {xdt} {M}x{N}x{K}")


def test_gemm_rowwise_back_to_back_calls_share_workspace(fp8bq):
    """Split tickets reset themselves: alternating shapes and codes on one
    workspace give the oracle's result every time."""
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    probs = [rowwise_problem(8, 1024, 2048, c, seed=i) + (c,)
             for i, c in enumerate(["e4m3", "int8", "e4m3"])]
    for rep in range(2):
        for (_, qa, sa, qw, sw, c) in probs:
            v = fp8bq.make_variant("swap", 16, 4 if rep == 0 else 0)
            o = fp8bq.fp8bq_gemm_rowwise(to_dev(qa), to_dev(sa), to_dev(qw), to_dev(sw), c,
                                         torch.bfloat16, workspace=ws, variant=v)
            torch.cuda.synchronize()
            check_gemm(o.float().cpu().numpy(), oracle.gemm_rowcol(qa, sa, qw, sw, CODES[c]),
                       "bf16", f"{c} rep {rep}")
    assert fp8bq.fp8bq_device_status() == 0
