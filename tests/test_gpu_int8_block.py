"""GPU parity of block INT8 (int8_w8a8, 1x128 activation groups, 128x128
weight blocks, fp32 scales; "vLLM 量化 Kernel 配置机制" §1) against the oracle:
quant codes and scales bit-exact; every GEMM kernel shape (warp-level int8
MMA: swap-AB token tiles 8..128; two e4m3 planes on the promotion kernel:
swap-AB and normal tiles; split-K, stream-K) on ragged shapes; DeepSeek-V3 shapes at full
size on sampled rows; the linear layer (quant + GEMM in one call)."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_group_gb300 import synth
from parity import TORCH_OUT, check_gemm, to_dev, to_dev_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8bq():
    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq as m
    return m


def f32_of_bf16(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("xdt", ["bf16", "fp16"])
@pytest.mark.parametrize("M,K", [(1, 128), (37, 1024), (64, 7168), (4096, 7168)])
def test_quant_act_int8_bit_exact(fp8bq, xdt, M, K):
    xb = synth.act_quant(M, K)  # spikes of +-1000 in every 8th row
    if xdt == "fp16":
        xb = synth.f32_to_f16_bits(f32_of_bf16(synth.act_decode(M, K)))
    x = to_dev_bits(xb, torch.bfloat16 if xdt == "bf16" else torch.float16)
    q, s = fp8bq.fp8bq_quant_act_int8(x)
    torch.cuda.synchronize()
    qo, so = oracle.quant_act_int8(xb, oracle.BF16 if xdt == "bf16" else oracle.FP16)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))  # incl. padding


@pytest.mark.parametrize("wdt", ["fp32", "bf16"])
@pytest.mark.parametrize("N,K", [(200, 256), (4096, 7168)])
def test_quant_weight_int8_bit_exact(fp8bq, wdt, N, K):
    if wdt == "fp32":
        w = synth.weight_f32(N, K)
        wd, code = to_dev(w), oracle.FP32
    else:
        w = synth.weight_bf16(N, K)
        wd, code = to_dev_bits(w), oracle.BF16
    q, s = fp8bq.fp8bq_quant_weight_int8(wd)
    torch.cuda.synchronize()
    qo, so = oracle.quant_weight_int8(w, code)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


def problem(M, N, K, seed=0, act=synth.act_prefill):
    xb = act(M, K, seed=seed)
    qa, sa = oracle.quant_act_int8(xb, oracle.BF16)
    qw, sw = oracle.quant_weight_int8(synth.weight_f32(N, K, seed=seed + 1), oracle.FP32)
    return xb, qa, sa, qw, sw


def run(fp8bq, qa, sa, qw, sw, out, variant=None):
    o = fp8bq.fp8bq_gemm_int8_block(to_dev(qa), to_dev(sa), to_dev(qw), to_dev(sw),
                                    TORCH_OUT[out], variant=variant)
    torch.cuda.synchronize()
    assert fp8bq.fp8bq_device_status() == 0
    return o.float().cpu().numpy()


VARIANTS = ([("swap", bn, 0) for bn in (8, 16, 32, 64, 128)] +
            [("swap", bn, 1) for bn in (16, 32, 64, 128)] +
            [("normal", bn, 1) for bn in (128, 256)])


@pytest.mark.parametrize("kind,bn,planes", VARIANTS)
@pytest.mark.parametrize("split", [1, 3, 0])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_gemm_int8_block_variants(fp8bq, kind, bn, planes, split, out):
    """planes=0: the warp-level int8 MMA with per-slab promotion; planes=1:
    the codes as two e4m3 planes on the tcgen05 FP8 MMA, promoted per slab
    on the CUDA cores.  Ragged: tokens past whole tiles, weight rows past a
    128-row block."""
    M, N, K = 150, 400, 1024
    _, qa, sa, qw, sw = problem(M, N, K, seed=bn + split)
    got = run(fp8bq, qa, sa, qw, sw, out, fp8bq.make_variant(kind, bn, split, 0, planes))
    check_gemm(got, oracle.gemm_int8_block(qa, sa, qw, sw), out,
               f"int8 block {kind}/{bn}/s{split}/planes={planes}")


@pytest.mark.parametrize("M,N,K", [(1, 1536, 1536), (8, 18432, 7168), (128, 7168, 18432),
                                   (2048, 4096, 7168)])
def test_gemm_int8_block_full_size_sampled(fp8bq, M, N, K):
    _, qa, sa, qw, sw = problem(M, N, K, seed=3)
    got = run(fp8bq, qa, sa, qw, sw, "bf16")
    for r in sorted({0, M // 2, M - 1}):
        ref = oracle.gemm_int8_block(qa, sa, qw, sw, rows=(r, 1))
        check_gemm(got[r:r + 1], ref, "bf16", f"int8 block {M}x{N}x{K} row {r}")


@pytest.mark.parametrize("xdt", ["bf16", "fp16"])
@pytest.mark.parametrize("M,N,K", [(5, 1536, 1536), (96, 4096, 7168)])
def test_linear_int8_block(fp8bq, xdt, M, N, K):
    xb = synth.act_decode(M, K, seed=11)
    if xdt == "fp16":
        xb = synth.f32_to_f16_bits(f32_of_bf16(xb))
    w = synth.weight_bf16(N, K)
    qw, sw = fp8bq.fp8bq_quant_weight_int8(to_dev_bits(w))
    x = to_dev_bits(xb, torch.bfloat16 if xdt == "bf16" else torch.float16)
    o = fp8bq.fp8bq_linear_int8_block(x, qw, sw, torch.bfloat16)
    torch.cuda.synchronize()
    assert fp8bq.fp8bq_device_status() == 0
    qa, sa = oracle.quant_act_int8(xb, oracle.BF16 if xdt == "bf16" else oracle.FP16)
    qwo, swo = oracle.quant_weight_int8(w, oracle.BF16)
    ref = oracle.gemm_int8_block(qa, sa, qwo, swo)
    check_gemm(o.float().cpu().numpy(), ref, "bf16", f"linear int8 block {xdt} {M}x{N}x{K}")
