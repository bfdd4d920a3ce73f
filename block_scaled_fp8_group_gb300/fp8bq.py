"""Thin Python binding of libfp8bq (the C ABI declared in include/fp8bq.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch supplies device memory and
streams); the functions have the same names as the C entry points.  If the
library has not been built, importing this module raises -- there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

LIB_PATH = _build.LIB

FP8BQ_OK = 0
STATUS_NAMES = {
    0: "FP8BQ_OK", 1: "FP8BQ_ERR_INVALID_ARG", 2: "FP8BQ_ERR_SHAPE", 3: "FP8BQ_ERR_ALIGNMENT",
    4: "FP8BQ_ERR_UNSUPPORTED", 5: "FP8BQ_ERR_WORKSPACE", 6: "FP8BQ_ERR_LAUNCH",
    7: "FP8BQ_ERR_DEVICE_TIMEOUT", 8: "FP8BQ_ERR_CUDA",
}
SCALE_FP32, SCALE_UE8M0 = 0, 1
CODE_E4M3, CODE_INT8 = 0, 1
BF16, FP16, FP32 = 0, 1, 2
KIND_NORMAL, KIND_SWAP_AB, KIND_SWAP_AB_64 = 0, 1, 2
_KIND_NAMES = {KIND_NORMAL: "normal", KIND_SWAP_AB: "swap", KIND_SWAP_AB_64: "swap64"}

EXPORTS = (
    "fp8bq_act_scale_bytes", "fp8bq_weight_scale_bytes", "fp8bq_gemm_workspace_bytes",
    "fp8bq_variant_workspace_bytes", "fp8bq_linear_workspace_bytes", "fp8bq_quant_act",
    "fp8bq_quant_weight", "fp8bq_gemm", "fp8bq_gemm_variant", "fp8bq_linear",
    "fp8bq_select_variant", "fp8bq_reload_table", "fp8bq_device_status",
    "fp8bq_selftest_wait_timeout", "fp8bq_status_string", "fp8bq_abi_version",
    "fp8bq_gemm_noalloc", "fp8bq_grouped_gemm", "fp8bq_grouped_gemm_variant",
    "fp8bq_select_grouped_variant", "fp8bq_grouped_gemm_workspace_bytes",
    "fp8bq_grouped_variant_workspace_bytes", "fp8bq_grouped_linear",
    "fp8bq_grouped_linear_workspace_bytes", "fp8bq_quant_rows", "fp8bq_gemm_rowwise",
    "fp8bq_gemm_rowwise_variant", "fp8bq_select_rowwise_variant",
    "fp8bq_rowwise_workspace_bytes", "fp8bq_rowwise_variant_workspace_bytes",
    "fp8bq_linear_rowwise", "fp8bq_linear_rowwise_workspace_bytes", "fp8bq_quant_act_int8",
    "fp8bq_quant_weight_int8", "fp8bq_gemm_int8_block", "fp8bq_gemm_int8_block_variant",
    "fp8bq_select_int8_block_variant", "fp8bq_int8_block_workspace_bytes",
    "fp8bq_int8_block_variant_workspace_bytes", "fp8bq_linear_int8_block",
    "fp8bq_linear_int8_block_workspace_bytes", "fp8bq_variant_supported",
)


class Fp8bqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({_lib.fp8bq_status_string(status).decode()})")


class Variant(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("block_n", ctypes.c_int32), ("split", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("from_table", ctypes.c_int32),
                ("mma_scale", ctypes.c_int32)]

    def as_dict(self):
        return {"kind": _KIND_NAMES.get(self.kind, str(self.kind)),
                "block_n": self.block_n, "split": self.split, "grid": self.grid,
                "mma_scale": self.mma_scale, "from_table": bool(self.from_table)}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libfp8bq.so is not built ({LIB_PATH}); run "
            "`python -m block_scaled_fp8_group_gb300.build` (needs nvcc) -- there is no fallback")
    lib = ctypes.CDLL(LIB_PATH)
    i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "fp8bq_act_scale_bytes": (sz, [i64, i64, i32, i32]),
        "fp8bq_weight_scale_bytes": (sz, [i64, i64, i32, i32]),
        "fp8bq_gemm_workspace_bytes": (sz, [i64, i64, i64, i32, i32]),
        "fp8bq_variant_workspace_bytes": (sz, [i64, i64, i64, ctypes.POINTER(Variant)]),
        "fp8bq_variant_supported": (i32, [i64, i64, i64, i32, ctypes.POINTER(Variant)]),
        "fp8bq_linear_workspace_bytes": (sz, [i64, i64, i64, i32, i32]),
        "fp8bq_quant_act": (i32, [vp, i32, i64, i64, i32, i32, vp, vp, vp]),
        "fp8bq_quant_weight": (i32, [vp, i32, i64, i64, i32, i32, i32, vp, vp, vp]),
        "fp8bq_gemm": (i32, [i64, i64, i64, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, sz,
                             vp]),
        "fp8bq_gemm_variant": (i32, [i64, i64, i64, vp, vp, vp, vp, i32, i32, vp,
                                     ctypes.POINTER(Variant), vp, sz, vp]),
        "fp8bq_linear": (i32, [vp, i32, i64, i64, i64, vp, vp, i32, i32, i32, i32, i32, vp, vp,
                               sz, vp]),
        "fp8bq_select_variant": (i32, [i64, i64, i64, i32, i32, ctypes.POINTER(Variant)]),
        "fp8bq_reload_table": (i32, []),
        "fp8bq_device_status": (i32, [ctypes.POINTER(ctypes.c_int), vp]),
        "fp8bq_selftest_wait_timeout": (i32, [ctypes.c_uint64, vp]),
        "fp8bq_gemm_noalloc": (i32, [i64, i64, i64, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                     vp]),
        "fp8bq_grouped_gemm": (i32, [i64, i64, i64, i64, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                     i32, vp, vp, sz, vp]),
        "fp8bq_grouped_gemm_variant": (i32, [i64, i64, i64, i64, vp, vp, vp, vp, vp, i32, i32,
                                             vp, ctypes.POINTER(Variant), vp, sz, vp]),
        "fp8bq_select_grouped_variant": (i32, [i64, i64, i64, i64, i32, i32,
                                               ctypes.POINTER(Variant)]),
        "fp8bq_grouped_gemm_workspace_bytes": (sz, [i64, i64, i64, i64, i32, i32]),
        "fp8bq_grouped_variant_workspace_bytes": (sz, [i64, i64, i64, i64,
                                                       ctypes.POINTER(Variant)]),
        "fp8bq_grouped_linear": (i32, [vp, i32, i64, i64, i64, i64, vp, vp, vp, i32, i32, i32,
                                       i32, i32, vp, vp, sz, vp]),
        "fp8bq_grouped_linear_workspace_bytes": (sz, [i64, i64, i64, i64, i32, i32]),
        "fp8bq_quant_rows": (i32, [vp, i32, i64, i64, i32, vp, vp, vp]),
        "fp8bq_gemm_rowwise": (i32, [i64, i64, i64, vp, vp, vp, vp, i32, i32, vp, vp, sz, vp]),
        "fp8bq_gemm_rowwise_variant": (i32, [i64, i64, i64, vp, vp, vp, vp, i32, i32, vp,
                                             ctypes.POINTER(Variant), vp, sz, vp]),
        "fp8bq_select_rowwise_variant": (i32, [i64, i64, i64, i32, i32,
                                               ctypes.POINTER(Variant)]),
        "fp8bq_rowwise_workspace_bytes": (sz, [i64, i64, i64, i32, i32]),
        "fp8bq_rowwise_variant_workspace_bytes": (sz, [i64, i64, i64, i32,
                                                       ctypes.POINTER(Variant)]),
        "fp8bq_linear_rowwise": (i32, [vp, i32, i64, i64, i64, vp, vp, i32, i32, vp, vp, sz,
                                       vp]),
        "fp8bq_linear_rowwise_workspace_bytes": (sz, [i64, i64, i64, i32, i32]),
        "fp8bq_quant_act_int8": (i32, [vp, i32, i64, i64, i32, vp, vp, vp]),
        "fp8bq_quant_weight_int8": (i32, [vp, i32, i64, i64, i32, i32, vp, vp, vp]),
        "fp8bq_gemm_int8_block": (i32, [i64, i64, i64, vp, vp, vp, vp, i32, i32, i32, i32, vp,
                                        vp, sz, vp]),
        "fp8bq_gemm_int8_block_variant": (i32, [i64, i64, i64, vp, vp, vp, vp, i32, vp,
                                                ctypes.POINTER(Variant), vp, sz, vp]),
        "fp8bq_select_int8_block_variant": (i32, [i64, i64, i64, i32, ctypes.POINTER(Variant)]),
        "fp8bq_int8_block_workspace_bytes": (sz, [i64, i64, i64, i32]),
        "fp8bq_int8_block_variant_workspace_bytes": (sz, [i64, i64, i64,
                                                          ctypes.POINTER(Variant)]),
        "fp8bq_linear_int8_block": (i32, [vp, i32, i64, i64, i64, vp, vp, i32, i32, i32, i32, vp,
                                          vp, sz, vp]),
        "fp8bq_linear_int8_block_workspace_bytes": (sz, [i64, i64, i64, i32]),
        "fp8bq_status_string": (ctypes.c_char_p, [i32]),
        "fp8bq_abi_version": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib():
    return _lib


# ------------------------------------------------------------------ helpers

def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        return {"fp32": SCALE_FP32, "ue8m0": SCALE_UE8M0}[fmt]
    return int(fmt)


_TORCH_TO_CODE = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}
_CODE_TO_TORCH = {v: k for k, v in _TORCH_TO_CODE.items()}


def _dtype_code(dt) -> int:
    if isinstance(dt, int):
        return dt
    if isinstance(dt, str):
        return {"bf16": BF16, "fp16": FP16, "fp32": FP32}[dt]
    return _TORCH_TO_CODE[dt]


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(st: int, where: str):
    if st != FP8BQ_OK:
        raise Fp8bqError(st, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


_ws_cache: dict = {}


def _workspace(nbytes: int, device) -> torch.Tensor | None:
    """A zero-filled per-device workspace, grown on demand.  The kernels leave
    it zero-filled, so it can be reused by calls that are ordered on the GPU;
    pass your own workspace for calls on concurrent streams."""
    if nbytes == 0:
        return None
    key = torch.device(device).index if torch.device(device).index is not None else \
        torch.cuda.current_device()
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


# ---------------------------------------------------------------- entry points

def fp8bq_act_scale_bytes(M: int, K: int, group: int = 128, fmt="fp32") -> int:
    return _lib.fp8bq_act_scale_bytes(M, K, group, _fmt(fmt))


def act_scale_shape(M: int, K: int, group: int = 128, fmt="fp32"):
    """(columns, Mp) of the activation scale buffer and its torch dtype."""
    G = K // group
    Mp = (M + 3) // 4 * 4
    if _fmt(fmt) == SCALE_UE8M0:
        return ((G + 3) // 4, Mp), torch.int32
    return (G, Mp), torch.float32


def fp8bq_quant_act(x: torch.Tensor, fmt="fp32", group: int = 128, q=None, s=None, stream=None):
    """x: [M,K] bf16/fp16 CUDA tensor -> (q uint8 [M,K], s fp32 [G,Mp] or int32 [ceil(G/4),Mp])."""
    _need(x, "x")
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if s is None:
        shape, dt = act_scale_shape(M, K, group, fmt)
        s = torch.empty(shape, dtype=dt, device=x.device)
    st = _lib.fp8bq_quant_act(_ptr(x), _dtype_code(x.dtype), M, K, group, _fmt(fmt), _ptr(q),
                              _ptr(s), _stream(stream))
    _check(st, "fp8bq_quant_act")
    return q, s


def fp8bq_quant_weight(w: torch.Tensor, fmt="fp32", block_n: int = 128, block_k: int = 128,
                       q=None, s=None, stream=None):
    """w: [N,K] fp32/bf16/fp16 -> (q uint8 [N,K], s fp32 [ceil(N/128), K/128])."""
    _need(w, "w")
    N, K = w.shape
    if q is None:
        q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty(((N + block_n - 1) // block_n, K // block_k), dtype=torch.float32,
                        device=w.device)
    st = _lib.fp8bq_quant_weight(_ptr(w), _dtype_code(w.dtype), N, K, block_n, block_k,
                                 _fmt(fmt), _ptr(q), _ptr(s), _stream(stream))
    _check(st, "fp8bq_quant_weight")
    return q, s


def fp8bq_select_variant(M: int, N: int, K: int, fmt="fp32", out_dtype=torch.bfloat16) -> dict:
    v = Variant()
    st = _lib.fp8bq_select_variant(M, N, K, _fmt(fmt), _dtype_code(out_dtype), ctypes.byref(v))
    _check(st, "fp8bq_select_variant")
    return v.as_dict()


def make_variant(kind, block_n: int, split: int = 1, grid: int = 0,
                 mma_scale: int = 0) -> Variant:
    """A GEMM variant; mma_scale=1 has the tensor core apply UE8M0 scales
    (block-scaled MMA; swap-AB, UE8M0, K % 512 == 0)."""
    k = kind if isinstance(kind, int) else {v: k for k, v in _KIND_NAMES.items()}[kind]
    return Variant(k, block_n, split, grid, 0, mma_scale)


def fp8bq_gemm_workspace_bytes(M, N, K, fmt="fp32", out_dtype=torch.bfloat16) -> int:
    return _lib.fp8bq_gemm_workspace_bytes(M, N, K, _fmt(fmt), _dtype_code(out_dtype))


def fp8bq_variant_supported(M, N, K, fmt, variant: Variant) -> bool:
    """Whether the kernels have this explicit shape for (M, N, K) and the scale
    format (host-only; launches nothing)."""
    return _lib.fp8bq_variant_supported(M, N, K, _fmt(fmt), ctypes.byref(variant)) == FP8BQ_OK


def fp8bq_variant_workspace_bytes(M, N, K, variant: Variant) -> int:
    return _lib.fp8bq_variant_workspace_bytes(M, N, K, ctypes.byref(variant))


def fp8bq_linear_workspace_bytes(M, N, K, fmt="fp32", out_dtype=torch.bfloat16) -> int:
    return _lib.fp8bq_linear_workspace_bytes(M, N, K, _fmt(fmt), _dtype_code(out_dtype))


def _out(M, N, out_dtype, device, out):
    if out is None:
        out = torch.empty((M, N), dtype=_CODE_TO_TORCH[_dtype_code(out_dtype)], device=device)
    return out


def fp8bq_gemm(a_q, a_s, w_q, w_s, fmt="fp32", out_dtype=torch.bfloat16, out=None,
               workspace=None, group: int = 128, block_n: int = 128, block_k: int = 128,
               stream=None):
    for t, n in ((a_q, "a_q"), (a_s, "a_s"), (w_q, "w_q"), (w_s, "w_s")):
        _need(t, n)
    M, K = a_q.shape
    N = w_q.shape[0]
    out = _out(M, N, out_dtype, a_q.device, out)
    nbytes = fp8bq_gemm_workspace_bytes(M, N, K, fmt, out_dtype)
    if workspace is None:
        workspace = _workspace(nbytes, a_q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.fp8bq_gemm(M, N, K, _ptr(a_q), _ptr(a_s), _ptr(w_q), _ptr(w_s), group, block_n,
                         block_k, _fmt(fmt), _dtype_code(out.dtype), _ptr(out), _ptr(workspace),
                         wsz, _stream(stream))
    _check(st, "fp8bq_gemm")
    return out


def fp8bq_gemm_variant(a_q, a_s, w_q, w_s, variant: Variant, fmt="fp32",
                       out_dtype=torch.bfloat16, out=None, workspace=None, stream=None):
    for t, n in ((a_q, "a_q"), (a_s, "a_s"), (w_q, "w_q"), (w_s, "w_s")):
        _need(t, n)
    M, K = a_q.shape
    N = w_q.shape[0]
    out = _out(M, N, out_dtype, a_q.device, out)
    nbytes = fp8bq_variant_workspace_bytes(M, N, K, variant)
    if workspace is None:
        workspace = _workspace(nbytes, a_q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.fp8bq_gemm_variant(M, N, K, _ptr(a_q), _ptr(a_s), _ptr(w_q), _ptr(w_s), _fmt(fmt),
                                 _dtype_code(out.dtype), _ptr(out), ctypes.byref(variant),
                                 _ptr(workspace), wsz, _stream(stream))
    _check(st, "fp8bq_gemm_variant")
    return out


def fp8bq_linear(x, w_q, w_s, fmt="ue8m0", out_dtype=torch.bfloat16, out=None, workspace=None,
                 group: int = 128, block_n: int = 128, block_k: int = 128, stream=None):
    """W8A8 linear layer: quantise x [M,K] (bf16/fp16) and multiply by the
    block-quantised weight.  The workspace holds the codes and scales."""
    for t, n in ((x, "x"), (w_q, "w_q"), (w_s, "w_s")):
        _need(t, n)
    M, K = x.shape
    N = w_q.shape[0]
    out = _out(M, N, out_dtype, x.device, out)
    nbytes = fp8bq_linear_workspace_bytes(M, N, K, fmt, out.dtype)
    if workspace is None:
        workspace = _workspace(nbytes, x.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.fp8bq_linear(_ptr(x), _dtype_code(x.dtype), M, N, K, _ptr(w_q), _ptr(w_s), group,
                           block_n, block_k, _fmt(fmt), _dtype_code(out.dtype), _ptr(out),
                           _ptr(workspace), wsz, _stream(stream))
    _check(st, "fp8bq_linear")
    return out


# ---------------------------------------------------------------- grouped GEMM

def fp8bq_select_grouped_variant(E: int, M_max: int, N: int, K: int, fmt="fp32",
                                 out_dtype=torch.bfloat16) -> dict:
    v = Variant()
    st = _lib.fp8bq_select_grouped_variant(E, M_max, N, K, _fmt(fmt), _dtype_code(out_dtype),
                                           ctypes.byref(v))
    _check(st, "fp8bq_select_grouped_variant")
    return v.as_dict()


def fp8bq_grouped_gemm_workspace_bytes(E, M_max, N, K, fmt="fp32", out_dtype=torch.bfloat16):
    return _lib.fp8bq_grouped_gemm_workspace_bytes(E, M_max, N, K, _fmt(fmt),
                                                   _dtype_code(out_dtype))


def fp8bq_grouped_variant_workspace_bytes(E, M_max, N, K, variant: Variant) -> int:
    return _lib.fp8bq_grouped_variant_workspace_bytes(E, M_max, N, K, ctypes.byref(variant))


def fp8bq_grouped_gemm(a_q, a_s, w_q, w_s, counts, fmt="fp32", out_dtype=torch.bfloat16,
                       out=None, workspace=None, variant: Variant | None = None, stream=None):
    """Grouped (MoE) GEMM, masked layout.  E = counts.numel() experts;
    a_q: [E*M_max, K] codes (a_s their scales); w_q: [E, N, K] (or [E*N, K])
    codes, w_s: [E, N/128, K/128] fp32; counts: int32 [E] on the GPU.  Rows of
    expert e at or past counts[e] of ``out`` [E*M_max, N] are left as they are."""
    for t, n in ((a_q, "a_q"), (a_s, "a_s"), (w_q, "w_q"), (w_s, "w_s"), (counts, "counts")):
        _need(t, n)
    if counts.dtype != torch.int32:
        raise ValueError("counts must be int32")
    E = counts.numel()
    rows, K = a_q.shape
    if E == 0 or rows % E:
        raise ValueError("a_q rows must be E * M_max")
    M_max = rows // E
    N = w_q.numel() // (E * K)
    out = _out(rows, N, out_dtype, a_q.device, out)
    if variant is None:
        nbytes = fp8bq_grouped_gemm_workspace_bytes(E, M_max, N, K, fmt, out.dtype)
    else:
        nbytes = fp8bq_grouped_variant_workspace_bytes(E, M_max, N, K, variant)
    if workspace is None:
        workspace = _workspace(nbytes, a_q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if variant is None:
        st = _lib.fp8bq_grouped_gemm(E, M_max, N, K, _ptr(counts), _ptr(a_q), _ptr(a_s),
                                     _ptr(w_q), _ptr(w_s), 128, 128, 128, _fmt(fmt),
                                     _dtype_code(out.dtype), _ptr(out), _ptr(workspace), wsz,
                                     _stream(stream))
        _check(st, "fp8bq_grouped_gemm")
    else:
        st = _lib.fp8bq_grouped_gemm_variant(E, M_max, N, K, _ptr(counts), _ptr(a_q), _ptr(a_s),
                                             _ptr(w_q), _ptr(w_s), _fmt(fmt),
                                             _dtype_code(out.dtype), _ptr(out),
                                             ctypes.byref(variant), _ptr(workspace), wsz,
                                             _stream(stream))
        _check(st, "fp8bq_grouped_gemm_variant")
    return out


def fp8bq_grouped_linear_workspace_bytes(E, M_max, N, K, fmt="ue8m0", out_dtype=torch.bfloat16):
    return _lib.fp8bq_grouped_linear_workspace_bytes(E, M_max, N, K, _fmt(fmt),
                                                     _dtype_code(out_dtype))


def fp8bq_grouped_linear(x, w_q, w_s, counts, fmt="ue8m0", out_dtype=torch.bfloat16, out=None,
                         workspace=None, stream=None):
    """Grouped W8A8 linear layer: quantise the experts' occupied rows of x
    [E*M_max, K] (bf16/fp16) and run the grouped GEMM with w_q [E, N, K],
    w_s [E, N/128, K/128]; counts int32 [E] on the GPU."""
    for t, n in ((x, "x"), (w_q, "w_q"), (w_s, "w_s"), (counts, "counts")):
        _need(t, n)
    if counts.dtype != torch.int32:
        raise ValueError("counts must be int32")
    E = counts.numel()
    rows, K = x.shape
    if E == 0 or rows % E:
        raise ValueError("x rows must be E * M_max")
    M_max = rows // E
    N = w_q.numel() // (E * K)
    out = _out(rows, N, out_dtype, x.device, out)
    nbytes = fp8bq_grouped_linear_workspace_bytes(E, M_max, N, K, fmt, out.dtype)
    if workspace is None:
        workspace = _workspace(nbytes, x.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.fp8bq_grouped_linear(_ptr(x), _dtype_code(x.dtype), E, M_max, N, K, _ptr(counts),
                                   _ptr(w_q), _ptr(w_s), 128, 128, 128, _fmt(fmt),
                                   _dtype_code(out.dtype), _ptr(out), _ptr(workspace), wsz,
                                   _stream(stream))
    _check(st, "fp8bq_grouped_linear")
    return out


# ------------------------------------------------ per-token x per-channel

def _code(code) -> int:
    if isinstance(code, str):
        return {"e4m3": CODE_E4M3, "int8": CODE_INT8}[code]
    return int(code)


def fp8bq_quant_rows(x: torch.Tensor, code="e4m3", q=None, s=None, stream=None):
    """One scale per row of x [R,K] (bf16/fp16/fp32): per-token activation or
    per-channel weight quant -> (q [R,K] uint8 e4m3 or int8 codes, s fp32 [R])."""
    _need(x, "x")
    R, K = x.shape
    if q is None:
        q = torch.empty((R, K), dtype=torch.int8 if _code(code) == CODE_INT8 else torch.uint8,
                        device=x.device)
    if s is None:
        s = torch.empty(R, dtype=torch.float32, device=x.device)
    st = _lib.fp8bq_quant_rows(_ptr(x), _dtype_code(x.dtype), R, K, _code(code), _ptr(q),
                               _ptr(s), _stream(stream))
    _check(st, "fp8bq_quant_rows")
    return q, s


def fp8bq_select_rowwise_variant(M: int, N: int, K: int, code="e4m3",
                                 out_dtype=torch.bfloat16) -> dict:
    v = Variant()
    st = _lib.fp8bq_select_rowwise_variant(M, N, K, _code(code), _dtype_code(out_dtype),
                                           ctypes.byref(v))
    _check(st, "fp8bq_select_rowwise_variant")
    return v.as_dict()


def fp8bq_rowwise_workspace_bytes(M, N, K, code="e4m3", out_dtype=torch.bfloat16) -> int:
    return _lib.fp8bq_rowwise_workspace_bytes(M, N, K, _code(code), _dtype_code(out_dtype))


def fp8bq_rowwise_variant_workspace_bytes(M, N, K, code, variant: Variant) -> int:
    return _lib.fp8bq_rowwise_variant_workspace_bytes(M, N, K, _code(code),
                                                      ctypes.byref(variant))


def fp8bq_gemm_rowwise(a_q, a_s, w_q, w_s, code="e4m3", out_dtype=torch.bfloat16, out=None,
                       workspace=None, variant: Variant | None = None, stream=None):
    """Rowwise-scaled GEMM: a_q [M,K] codes, a_s fp32 [M]; w_q [N,K], w_s fp32 [N]."""
    for t, n in ((a_q, "a_q"), (a_s, "a_s"), (w_q, "w_q"), (w_s, "w_s")):
        _need(t, n)
    M, K = a_q.shape
    N = w_q.shape[0]
    out = _out(M, N, out_dtype, a_q.device, out)
    if variant is None:
        nbytes = fp8bq_rowwise_workspace_bytes(M, N, K, code, out.dtype)
    else:
        nbytes = fp8bq_rowwise_variant_workspace_bytes(M, N, K, code, variant)
    if workspace is None:
        workspace = _workspace(nbytes, a_q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if variant is None:
        st = _lib.fp8bq_gemm_rowwise(M, N, K, _ptr(a_q), _ptr(a_s), _ptr(w_q), _ptr(w_s),
                                     _code(code), _dtype_code(out.dtype), _ptr(out),
                                     _ptr(workspace), wsz, _stream(stream))
    else:
        st = _lib.fp8bq_gemm_rowwise_variant(M, N, K, _ptr(a_q), _ptr(a_s), _ptr(w_q),
                                             _ptr(w_s), _code(code), _dtype_code(out.dtype),
                                             _ptr(out), ctypes.byref(variant), _ptr(workspace),
                                             wsz, _stream(stream))
    _check(st, "fp8bq_gemm_rowwise")
    return out


def fp8bq_linear_rowwise_workspace_bytes(M, N, K, code="e4m3", out_dtype=torch.bfloat16):
    return _lib.fp8bq_linear_rowwise_workspace_bytes(M, N, K, _code(code), _dtype_code(out_dtype))


def fp8bq_linear_rowwise(x, w_q, w_s, code="e4m3", out_dtype=torch.bfloat16, out=None,
                         workspace=None, stream=None):
    """Rowwise W8A8 linear layer: per-token quant of x [M,K] (bf16/fp16) and
    the rowwise GEMM with w_q [N,K], w_s fp32 [N], in one call."""
    for t, n in ((x, "x"), (w_q, "w_q"), (w_s, "w_s")):
        _need(t, n)
    M, K = x.shape
    N = w_q.shape[0]
    out = _out(M, N, out_dtype, x.device, out)
    nbytes = fp8bq_linear_rowwise_workspace_bytes(M, N, K, code, out.dtype)
    if workspace is None:
        workspace = _workspace(nbytes, x.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.fp8bq_linear_rowwise(_ptr(x), _dtype_code(x.dtype), M, N, K, _ptr(w_q), _ptr(w_s),
                                   _code(code), _dtype_code(out.dtype), _ptr(out),
                                   _ptr(workspace), wsz, _stream(stream))
    _check(st, "fp8bq_linear_rowwise")
    return out


# ------------------------------------------------------------------ block INT8

def fp8bq_quant_act_int8(x: torch.Tensor, group: int = 128, q=None, s=None, stream=None):
    """x [M,K] bf16/fp16 -> (q int8 [M,K], s fp32 [K/128, Mp] column-major)."""
    _need(x, "x")
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if s is None:
        s = torch.empty(act_scale_shape(M, K, group, "fp32")[0], dtype=torch.float32,
                        device=x.device)
    st = _lib.fp8bq_quant_act_int8(_ptr(x), _dtype_code(x.dtype), M, K, group, _ptr(q), _ptr(s),
                                   _stream(stream))
    _check(st, "fp8bq_quant_act_int8")
    return q, s


def fp8bq_quant_weight_int8(w: torch.Tensor, block_n: int = 128, block_k: int = 128, q=None,
                            s=None, stream=None):
    """w [N,K] fp32/bf16/fp16 -> (q int8 [N,K], s fp32 [ceil(N/128), K/128])."""
    _need(w, "w")
    N, K = w.shape
    if q is None:
        q = torch.empty((N, K), dtype=torch.int8, device=w.device)
    if s is None:
        s = torch.empty(((N + block_n - 1) // block_n, K // block_k), dtype=torch.float32,
                        device=w.device)
    st = _lib.fp8bq_quant_weight_int8(_ptr(w), _dtype_code(w.dtype), N, K, block_n, block_k,
                                      _ptr(q), _ptr(s), _stream(stream))
    _check(st, "fp8bq_quant_weight_int8")
    return q, s


def fp8bq_select_int8_block_variant(M, N, K, out_dtype=torch.bfloat16) -> dict:
    v = Variant()
    st = _lib.fp8bq_select_int8_block_variant(M, N, K, _dtype_code(out_dtype), ctypes.byref(v))
    _check(st, "fp8bq_select_int8_block_variant")
    return v.as_dict()


def fp8bq_gemm_int8_block(a_q, a_s, w_q, w_s, out_dtype=torch.bfloat16, out=None,
                          workspace=None, variant: Variant | None = None, stream=None):
    """Block INT8 GEMM: int8 codes with fp32 1x128 activation-group and 128x128
    weight-block scales."""
    for t, n in ((a_q, "a_q"), (a_s, "a_s"), (w_q, "w_q"), (w_s, "w_s")):
        _need(t, n)
    M, K = a_q.shape
    N = w_q.shape[0]
    out = _out(M, N, out_dtype, a_q.device, out)
    if variant is None:
        nbytes = _lib.fp8bq_int8_block_workspace_bytes(M, N, K, _dtype_code(out.dtype))
    else:
        nbytes = _lib.fp8bq_int8_block_variant_workspace_bytes(M, N, K, ctypes.byref(variant))
    if workspace is None:
        workspace = _workspace(nbytes, a_q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if variant is None:
        st = _lib.fp8bq_gemm_int8_block(M, N, K, _ptr(a_q), _ptr(a_s), _ptr(w_q), _ptr(w_s), 128,
                                        128, 128, _dtype_code(out.dtype), _ptr(out),
                                        _ptr(workspace), wsz, _stream(stream))
    else:
        st = _lib.fp8bq_gemm_int8_block_variant(M, N, K, _ptr(a_q), _ptr(a_s), _ptr(w_q),
                                                _ptr(w_s), _dtype_code(out.dtype), _ptr(out),
                                                ctypes.byref(variant), _ptr(workspace), wsz,
                                                _stream(stream))
    _check(st, "fp8bq_gemm_int8_block")
    return out


def fp8bq_linear_int8_block(x, w_q, w_s, out_dtype=torch.bfloat16, out=None, workspace=None,
                            stream=None):
    """Block INT8 linear layer: int8 group quant of x [M,K] (bf16/fp16), then
    the block INT8 GEMM, in one call."""
    for t, n in ((x, "x"), (w_q, "w_q"), (w_s, "w_s")):
        _need(t, n)
    M, K = x.shape
    N = w_q.shape[0]
    out = _out(M, N, out_dtype, x.device, out)
    nbytes = _lib.fp8bq_linear_int8_block_workspace_bytes(M, N, K, _dtype_code(out.dtype))
    if workspace is None:
        workspace = _workspace(nbytes, x.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.fp8bq_linear_int8_block(_ptr(x), _dtype_code(x.dtype), M, N, K, _ptr(w_q),
                                      _ptr(w_s), 128, 128, 128, _dtype_code(out.dtype), _ptr(out),
                                      _ptr(workspace), wsz, _stream(stream))
    _check(st, "fp8bq_linear_int8_block")
    return out


def fp8bq_device_status(stream=None) -> int:
    code = ctypes.c_int(0)
    st = _lib.fp8bq_device_status(ctypes.byref(code), _stream(stream))
    _check(st, "fp8bq_device_status")
    return code.value


def fp8bq_selftest_wait_timeout(timeout_ns: int, stream=None):
    _check(_lib.fp8bq_selftest_wait_timeout(timeout_ns, _stream(stream)),
           "fp8bq_selftest_wait_timeout")


def fp8bq_reload_table():
    _check(_lib.fp8bq_reload_table(), "fp8bq_reload_table")
