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
    # the selected kernel splits K, so the shared array is really used (and
    # the second call finds it as the first one left it)
    assert 0 < need <= SCRATCH_BYTES
    ref = fp8bq.fp8bq_gemm(aq, as_, wq, ws, fmt=fmt, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(fp8bq, aq, as_, wq, ws, fmt, out) == 0
        torch.cuda.synchronize()
        # the same kernel on the same inputs with a fixed-order split
        # reduction: the result equals fp8bq_gemm's bit for bit (and so lies
        # within the GEMM tolerance of the oracle that fp8bq_gemm's own tests
        # check)
        assert torch.equal(out, ref), f"noalloc call {call} differs from fp8bq_gemm"
        check_gemm(out.float().cpu().numpy(), ref64, "bf16", f"noalloc call {call}")
    assert fp8bq.fp8bq_device_status() == 0


# Shapes whose table-selected kernel (a stream-K schedule over 256-wide tiles)
# needs more than the 32 MiB array; the test uses the first that does.
OVERSIZED = [(1536, 4096, 7168, "fp32"), (2048, 4096, 7168, "fp32"), (4096, 4096, 7168, "fp32"),
             (1536, 4096, 7168, "ue8m0"), (1024, 7168, 18432, "fp32"),
             (2048, 7168, 18432, "ue8m0"), (256, 4096, 7168, "fp32")]


def test_noalloc_rejects_problems_beyond_the_scratch(fp8bq):
    found = [(M, N, K, fmt) for (M, N, K, fmt) in OVERSIZED
             if fp8bq.fp8bq_gemm_workspace_bytes(M, N, K, fmt, torch.bfloat16) > SCRATCH_BYTES]
    assert found, "no candidate shape needs more than 32 MiB under the current table"
    M, N, K, fmt = found[0]
    aq = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    shape, dt = fp8bq.act_scale_shape(M, K, 128, fmt)
    as_ = torch.zeros(shape, dtype=dt, device="cuda")
    wq = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    ws = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(fp8bq, aq, as_, wq, ws, fmt, out) == 5  # FP8BQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    # rejected on the host before any launch: the output is untouched
    assert bool((out == 7.0).all())
