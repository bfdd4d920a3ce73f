"""fp8bq_gemm_noalloc: the GEMM for callers that cannot allocate device memory
(runtimes that own all device memory from start-up, code that must not risk
an allocation's device synchronisation, plug-ins that only get tensors and a
stream).  It uses a scratch array built into the library instead of a
caller-provided workspace.  Called through the C ABI and compared with
fp8bq_gemm on the same inputs, twice in a row (the second call finds the
shared array as the first one left it).

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_fp8_group_gb300 import synth
from parity import check_gemm

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def fp8bq():
    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq as m
    return m


def problem(fp8bq, M, N, K, fmt):
    x = torch.from_numpy(synth.act_decode(M, K).view(np.int16)).view(torch.bfloat16).cuda()
    w = torch.from_numpy(synth.weight_bf16(N, K).view(np.int16)).view(torch.bfloat16).cuda()
    wq, ws = fp8bq.fp8bq_quant_weight(w, fmt)
    aq, as_ = fp8bq.fp8bq_quant_act(x, fmt)
    return aq, as_, wq, ws


def call_noalloc(fp8bq, aq, as_, wq, ws, fmt, out):
    M, K = aq.shape
    N = wq.shape[0]
    st = fp8bq.lib().fp8bq_gemm_noalloc(
        M, N, K, aq.data_ptr(), as_.data_ptr(), wq.data_ptr(), ws.data_ptr(), 128, 128, 128,
        1 if fmt == "ue8m0" else 0, 0, out.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.parametrize("M,N,K,fmt", [(8, 4096, 7168, "ue8m0"), (16, 1536, 1536, "fp32"),
                                       (24, 7168, 18432, "ue8m0"), (3, 384, 1280, "fp32")])
def test_noalloc_matches_gemm_twice(fp8bq, M, N, K, fmt):
    aq, as_, wq, ws = problem(fp8bq, M, N, K, fmt)
    need = fp8bq.fp8bq_gemm_workspace_bytes(M, N, K, fmt, torch.bfloat16)
    assert need <= SCRATCH_BYTES
    ref = fp8bq.fp8bq_gemm(aq, as_, wq, ws, fmt=fmt, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(fp8bq, aq, as_, wq, ws, fmt, out) == 0
        torch.cuda.synchronize()
        check_gemm(out.float().cpu().numpy(), ref64, "bf16", f"noalloc call {call}")
    assert fp8bq.fp8bq_device_status() == 0


def test_noalloc_rejects_problems_beyond_the_scratch(fp8bq):
    # a large split problem (default variant: stream-K over 256-wide tiles)
    M, N, K = 256, 4096, 7168
    need = fp8bq.fp8bq_gemm_workspace_bytes(M, N, K, "fp32", torch.bfloat16)
    if need <= SCRATCH_BYTES:
        pytest.skip("the selected kernel for this shape fits the scratch")
    aq = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    as_ = torch.ones((K // 128, M), dtype=torch.float32, device="cuda")
    wq = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    ws = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(fp8bq, aq, as_, wq, ws, "fp32", out) == 5  # FP8BQ_ERR_WORKSPACE
