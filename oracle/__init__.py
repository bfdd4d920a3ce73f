"""CPU oracle of the W8A8 block-FP8 linear path (ctypes binding of oracle.c).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the benchmark's ``cpu_baseline`` / ``--impl reference`` legs.  The product
package never imports it, and it shares no code with the CUDA path.

Every function takes and returns numpy arrays; the C source states which page
and section each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

BF16, FP16, FP32 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, no CUDA)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        return _LIB
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        l.oracle_e4m3_decode.restype = dp
        l.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        l.oracle_e4m3_encode.restype = ctypes.c_uint8
        l.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        l.oracle_bf16_to_f32.restype = ctypes.c_float
        l.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        l.oracle_f16_to_f32.restype = ctypes.c_float
        l.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        l.oracle_group_scale.restype = ctypes.c_float
        l.oracle_group_scale.argtypes = [ctypes.c_float, i32]
        l.oracle_quant_value.restype = ctypes.c_uint8
        l.oracle_quant_value.argtypes = [ctypes.c_float, ctypes.c_float]
        l.oracle_act_scale_bytes.restype = i64
        l.oracle_act_scale_bytes.argtypes = [i64, i64, i32, i32]
        l.oracle_quant_act.restype = i32
        l.oracle_quant_act.argtypes = [vp, i32, i64, i64, i32, i32, vp, vp]
        l.oracle_quant_weight.restype = i32
        l.oracle_quant_weight.argtypes = [vp, i32, i64, i64, i32, i32, i32, vp, vp]
        l.oracle_act_scale.restype = dp
        l.oracle_act_scale.argtypes = [vp, i32, i64, i64, i32, i64, i64]
        l.oracle_gemm.restype = i32
        l.oracle_gemm.argtypes = [i64, i64, i64, vp, vp, i32, vp, vp, i32, i32, i32, i64, i64, vp]
        l.oracle_gemm_elem.restype = dp
        l.oracle_gemm_elem.argtypes = [i64, i64, i64, vp, vp, i32, vp, vp, i32, i32, i32, i64, i64]
        l.oracle_quant_rows.restype = i32
        l.oracle_quant_rows.argtypes = [vp, i32, i64, i64, i32, vp, vp]
        l.oracle_int8_value.restype = ctypes.c_int8
        l.oracle_int8_value.argtypes = [ctypes.c_float, ctypes.c_float]
        l.oracle_gemm_rowcol.restype = i32
        l.oracle_gemm_rowcol.argtypes = [i64, i64, i64, vp, vp, vp, vp, i32, i64, i64, vp]
        l.oracle_quant_act_int8.restype = i32
        l.oracle_quant_act_int8.argtypes = [vp, i32, i64, i64, i32, vp, vp]
        l.oracle_quant_weight_int8.restype = i32
        l.oracle_quant_weight_int8.argtypes = [vp, i32, i64, i64, i32, i32, vp, vp]
        l.oracle_gemm_int8_block.restype = i32
        l.oracle_gemm_int8_block.argtypes = [i64, i64, i64, vp, vp, vp, vp, i32, i32, i32, i64,
                                             i64, vp]
        l.oracle_calc_diff.restype = dp
        l.oracle_calc_diff.argtypes = [vp, vp, i64]
        _lib = l
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ------------------------------------------------------------------ codecs --

def e4m3_decode(code: int) -> float:
    return lib().oracle_e4m3_decode(int(code))


def e4m3_decode_all() -> np.ndarray:
    """Decoded value of all 256 codes (NaN for 0x7F, 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(y: float) -> int:
    return int(lib().oracle_e4m3_encode(float(y)))


def group_scale(amax: float, ue8m0: bool) -> np.float32:
    return np.float32(lib().oracle_group_scale(float(amax), int(bool(ue8m0))))


def quant_value(x: float, s: float) -> int:
    return int(lib().oracle_quant_value(float(x), float(s)))


def bf16_to_f32(bits: int) -> np.float32:
    return np.float32(lib().oracle_bf16_to_f32(int(bits)))


def f16_to_f32(bits: int) -> np.float32:
    return np.float32(lib().oracle_f16_to_f32(int(bits)))


# ------------------------------------------------------------------- quant --

def act_scale_bytes(M: int, K: int, group: int, ue8m0: bool) -> int:
    return int(lib().oracle_act_scale_bytes(M, K, group, int(bool(ue8m0))))


def quant_act(x_bits: np.ndarray, x_dtype: int, group: int, ue8m0: bool):
    """x_bits: uint16 [M,K] (bf16 or fp16 bit patterns).

    Returns (q uint8 [M,K], s) with s float32 [G, Mp] (fp32 mode) or uint32
    [ceil(G/4), Mp] (UE8M0 packed mode), both column-major in the sense
    that a group's scales for consecutive rows are contiguous.
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    G = K // group
    Mp = (M + 3) // 4 * 4
    q = np.empty((M, K), dtype=np.uint8)
    if ue8m0:
        s = np.empty(((G + 3) // 4, Mp), dtype=np.uint32)
    else:
        s = np.empty((G, Mp), dtype=np.float32)
    rc = lib().oracle_quant_act(_ptr(x_bits), x_dtype, M, K, group, int(bool(ue8m0)),
                                _ptr(q), _ptr(s))
    if rc != 0:
        raise ValueError("oracle_quant_act: bad arguments")
    return q, s


def quant_weight(w: np.ndarray, w_dtype: int, bn: int = 128, bk: int = 128, ue8m0: bool = False):
    """w: [N,K] float32 (w_dtype FP32) or uint16 bit patterns (BF16/FP16)."""
    w = np.ascontiguousarray(w)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty(((N + bn - 1) // bn, K // bk), dtype=np.float32)
    rc = lib().oracle_quant_weight(_ptr(w), w_dtype, N, K, bn, bk, int(bool(ue8m0)),
                                   _ptr(q), _ptr(s))
    if rc != 0:
        raise ValueError("oracle_quant_weight: bad arguments")
    return q, s


def act_scale(s: np.ndarray, ue8m0: bool, M: int, K: int, group: int, m: int, g: int) -> float:
    return lib().oracle_act_scale(_ptr(s), int(bool(ue8m0)), M, K, group, m, g)


# -------------------------------------------------------------------- GEMM --

def gemm(qa, sa, qw, sw, ue8m0: bool, group: int = 128, bn: int = 128, bk: int = 128,
         rows=None) -> np.ndarray:
    """fp64 reference [M,N] (or the row range ``rows=(row0, count)``)."""
    M, K = qa.shape
    N = qw.shape[0]
    row0, cnt = (0, M) if rows is None else rows
    out = np.empty((cnt, N), dtype=np.float64)
    rc = lib().oracle_gemm(M, N, K, _ptr(qa), _ptr(sa), int(bool(ue8m0)), _ptr(qw), _ptr(sw),
                           group, bn, bk, row0, cnt, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_gemm: bad arguments")
    return out


def gemm_elem(qa, sa, qw, sw, ue8m0: bool, m: int, n: int, group: int = 128, bn: int = 128,
              bk: int = 128) -> float:
    M, K = qa.shape
    N = qw.shape[0]
    return lib().oracle_gemm_elem(M, N, K, _ptr(qa), _ptr(sa), int(bool(ue8m0)), _ptr(qw),
                                  _ptr(sw), group, bn, bk, m, n)


def grouped_gemm(qa, sa, qw, sw, counts, ue8m0: bool, out=None, group: int = 128,
                 bn: int = 128, bk: int = 128) -> np.ndarray:
    """Grouped (MoE) GEMM, masked layout: E = len(counts) experts; expert e
    owns token rows [e*M_max, e*M_max + c_e) of qa (c_e = counts[e] clamped
    to [0, M_max]) and weights qw[e] [N,K] with scales sw[e].  Each expert's
    rows are the plain block-scaled GEMM of those rows and its own weights
    ("vLLM 量化 Kernel 配置机制" §5 applies the linear path's kernel scheme to
    MoE experts; the per-expert product is "vLLM DeepGEMM FP8 Block GEMM
    基准测试" §4.2's fp8_gemm_nt).  Rows past an expert's count keep the
    value they have in ``out`` (NaN when out is None).

    qa [E*M_max, K] codes, sa their scales in the quant layout of all
    E*M_max rows; qw [E, N, K]; sw [E, ceil(N/128), K/128]."""
    counts = np.asarray(counts)
    E = counts.shape[0]
    rows, K = qa.shape
    M_max = rows // E
    N = qw.shape[1]
    if out is None:
        out = np.full((rows, N), np.nan)
    for e in range(E):
        c = int(min(max(int(counts[e]), 0), M_max))
        if c == 0:
            continue
        # the plain GEMM over all rows' scales, restricted to this expert's
        # rows and weights
        out[e * M_max:e * M_max + c] = gemm(qa, sa, np.ascontiguousarray(qw[e]),
                                            np.ascontiguousarray(sw[e]), ue8m0, group, bn, bk,
                                            rows=(e * M_max, c))
    return out


# ---------------------------------------------- per-token x per-channel --

def quant_rows(x: np.ndarray, x_dtype: int, int8: bool = False):
    """One scale per row ("用 Helion 为 vLLM 构建高性能可移植线性后端", 范围:
    FP8_Dynamic and W8A8_INT8 use per-token activation and per-channel weight
    scales).  x: [R,K] float32 (FP32) or uint16 bit patterns (BF16/FP16).
    Returns (q [R,K]: uint8 e4m3 codes, or int8 when int8=True; s float32 [R])."""
    x = np.ascontiguousarray(x)
    R, K = x.shape
    q = np.empty((R, K), dtype=np.int8 if int8 else np.uint8)
    s = np.empty(R, dtype=np.float32)
    rc = lib().oracle_quant_rows(_ptr(x), x_dtype, R, K, int(bool(int8)), _ptr(q), _ptr(s))
    if rc != 0:
        raise ValueError("oracle_quant_rows: bad arguments")
    return q, s


def int8_value(x: float, s: float) -> int:
    return int(lib().oracle_int8_value(float(x), float(s)))


def gemm_rowcol(qa, sa, qw, sw, int8: bool = False, rows=None) -> np.ndarray:
    """fp64 reference of the per-token x per-channel GEMM:
    (sa[m] * sw[n]) * sum_k dec(qa[m,k]) * dec(qw[n,k]); rows=(row0, count)."""
    qa = np.ascontiguousarray(qa)
    qw = np.ascontiguousarray(qw)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    row0, cnt = (0, M) if rows is None else rows
    out = np.empty((cnt, N), dtype=np.float64)
    rc = lib().oracle_gemm_rowcol(M, N, K, _ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw),
                                  int(bool(int8)), row0, cnt, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_gemm_rowcol: bad arguments")
    return out


# ------------------------------------------------------------ block INT8 --

def quant_act_int8(x_bits: np.ndarray, x_dtype: int, group: int = 128):
    """Per-token-group quant with int8 codes ("vLLM 量化 Kernel 配置机制" §1,
    int8_w8a8 with block_shape [128,128]).  Returns (q int8 [M,K], s float32
    [G, Mp] column-major as quant_act's fp32 mode)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    G, Mp = K // group, (M + 3) // 4 * 4
    q = np.empty((M, K), dtype=np.int8)
    s = np.empty((G, Mp), dtype=np.float32)
    rc = lib().oracle_quant_act_int8(_ptr(x_bits), x_dtype, M, K, group, _ptr(q), _ptr(s))
    if rc != 0:
        raise ValueError("oracle_quant_act_int8: bad arguments")
    return q, s


def quant_weight_int8(w: np.ndarray, w_dtype: int, bn: int = 128, bk: int = 128):
    w = np.ascontiguousarray(w)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.int8)
    s = np.empty(((N + bn - 1) // bn, K // bk), dtype=np.float32)
    rc = lib().oracle_quant_weight_int8(_ptr(w), w_dtype, N, K, bn, bk, _ptr(q), _ptr(s))
    if rc != 0:
        raise ValueError("oracle_quant_weight_int8: bad arguments")
    return q, s


def gemm_int8_block(qa, sa, qw, sw, group: int = 128, bn: int = 128, bk: int = 128,
                    rows=None) -> np.ndarray:
    """fp64 reference of the block INT8 GEMM: every K slab's exact integer sum
    promoted by sa[m,kb] * sw[n/bn,kb], accumulated in slab order."""
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    row0, cnt = (0, M) if rows is None else rows
    out = np.empty((cnt, N), dtype=np.float64)
    rc = lib().oracle_gemm_int8_block(M, N, K, _ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), group,
                                      bn, bk, row0, cnt, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_gemm_int8_block: bad arguments")
    return out


def calc_diff(x: np.ndarray, y: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float64).ravel()
    y = np.ascontiguousarray(y, dtype=np.float64).ravel()
    return lib().oracle_calc_diff(_ptr(x), _ptr(y), x.size)
