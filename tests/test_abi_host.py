"""Host-side checks of the C ABI (no GPU needed, no compute launched).

* the library loads and exports every function include/fp8bq.h declares;
* size queries agree with the oracle's layout arithmetic;
* invalid arguments are rejected on the host with the documented status;
* the per-shape table lookup: nearest M, ties to the smaller grid point
  ("vLLM 量化 Kernel 配置机制" §4.2 worked examples M=37 -> 32, M=2050 -> 2048),
  a missing entry falls back to the default variant.
"""
import ctypes
import os
import re

import pytest

import oracle
from block_scaled_fp8_group_gb300 import build, fp8bq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def header_functions():
    text = open(os.path.join(ROOT, "include", "fp8bq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8bq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 15
    lib = ctypes.CDLL(fp8bq.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(fp8bq.EXPORTS)


def test_abi_version_and_status_strings():
    lib = fp8bq.lib()
    assert lib.fp8bq_abi_version() == 1
    for code in range(9):
        assert lib.fp8bq_status_string(code)


@pytest.mark.parametrize("M,K", [(1, 128), (3, 640), (16, 1536), (37, 7168), (1025, 18432)])
@pytest.mark.parametrize("ue", [False, True])
def test_act_scale_bytes_matches_oracle(M, K, ue):
    assert fp8bq.fp8bq_act_scale_bytes(M, K, 128, "ue8m0" if ue else "fp32") == \
        oracle.act_scale_bytes(M, K, 128, ue)


def test_size_queries_reject_bad_shapes():
    lib = fp8bq.lib()
    assert lib.fp8bq_act_scale_bytes(4, 100, 128, 0) == 0
    assert lib.fp8bq_act_scale_bytes(4, 256, 64, 0) == 0
    assert lib.fp8bq_weight_scale_bytes(200, 384, 128, 128) == 4 * 2 * 3
    assert lib.fp8bq_weight_scale_bytes(200, 384, 64, 128) == 0


def call_gemm(M=16, N=128, K=256, ptr=4096, group=128, fmt=0, out=0, ws=None, wsb=0):
    lib = fp8bq.lib()
    p = ctypes.c_void_p(ptr)
    return lib.fp8bq_gemm(M, N, K, p, p, p, p, group, 128, 128, fmt, out, p, ws, wsb, None)


def test_gemm_argument_errors_on_host():
    assert call_gemm(K=100) == 2          # K % 128
    assert call_gemm(K=0) == 2            # K == 0
    assert call_gemm(N=100) == 2          # N % 64
    assert call_gemm(M=-1) == 1
    assert call_gemm(fmt=7) == 1
    assert call_gemm(out=9) == 1
    assert call_gemm(group=64) == 4
    assert call_gemm(ptr=4100) == 3       # not 16-byte aligned
    assert call_gemm(ptr=0) == 1          # null
    assert call_gemm(M=0) == 0            # empty: no-op
    assert call_gemm(N=0) == 0


def test_quant_argument_errors_on_host():
    lib = fp8bq.lib()
    p = ctypes.c_void_p(4096)
    assert lib.fp8bq_quant_act(p, 0, 4, 100, 128, 0, p, p, None) == 2
    assert lib.fp8bq_quant_act(p, 2, 4, 128, 128, 0, p, p, None) == 4   # fp32 input
    assert lib.fp8bq_quant_act(p, 0, 4, 128, 32, 0, p, p, None) == 4
    assert lib.fp8bq_quant_act(ctypes.c_void_p(4104), 0, 4, 128, 128, 0, p, p, None) == 3
    assert lib.fp8bq_quant_act(p, 0, 0, 128, 128, 0, p, p, None) == 0
    assert lib.fp8bq_quant_weight(p, 0, 4, 128, 128, 64, 0, p, p, None) == 4
    assert lib.fp8bq_quant_weight(p, 0, 4, 120, 128, 128, 0, p, p, None) == 2


def test_linear_argument_errors_on_host():
    lib = fp8bq.lib()
    p = ctypes.c_void_p(4096)
    # workspace not 256-byte aligned
    assert lib.fp8bq_linear(p, 0, 4, 128, 128, p, p, 128, 128, 128, 1, 0, p,
                            ctypes.c_void_p(4096 + 16), 1 << 20, None) == 5
    assert lib.fp8bq_linear(p, 2, 4, 128, 128, p, p, 128, 128, 128, 1, 0, p, p, 1 << 20,
                            None) == 4


@pytest.fixture()
def fake_table(tmp_path, monkeypatch):
    t = tmp_path / "t.tbl"
    t.write_text(
        "# N K fmt out M kind block_n split grid\n"
        "4096 7168 ue8m0 bf16 1 swap 16 4 0\n"
        "4096 7168 ue8m0 bf16 8 swap 16 4 0 1\n"
        "4096 7168 ue8m0 bf16 32 swap 32 2 0\n"
        "4096 7168 ue8m0 bf16 64 swap 64 1 120\n"
        "4096 7168 ue8m0 bf16 2048 normal 256 1 0\n"
        "4096 7168 ue8m0 bf16 4096 normal 128 1 0\n"
        "this line is malformed and skipped\n")
    monkeypatch.setenv("FP8BQ_TABLE", str(t))
    fp8bq.fp8bq_reload_table()
    yield
    monkeypatch.delenv("FP8BQ_TABLE")
    fp8bq.fp8bq_reload_table()


def test_nearest_m_lookup(fake_table):
    sel = lambda M: fp8bq.fp8bq_select_variant(M, 4096, 7168, "ue8m0", "bf16")
    assert sel(37)["block_n"] == 32          # 37 -> 32
    assert sel(2050)["block_n"] == 256       # 2050 -> 2048
    assert sel(48)["block_n"] == 32          # tie between 32 and 64 -> smaller
    v = sel(64)
    assert v == {"kind": "swap", "block_n": 64, "split": 1, "grid": 120, "mma_scale": 0,
                 "from_table": True}
    assert sel(1)["split"] == 4 and sel(1)["mma_scale"] == 0  # 9-column line
    assert sel(8)["split"] == 4 and sel(8)["mma_scale"] == 1  # optional 10th column
    assert sel(10 ** 6)["block_n"] == 128    # beyond the grid -> largest key
    assert sel(3072)["block_n"] == 256       # tie 2048/4096 -> smaller


def test_table_miss_uses_default(fake_table):
    v = fp8bq.fp8bq_select_variant(8, 7168, 18432, "ue8m0", "bf16")
    assert v["from_table"] is False and v["kind"] == "swap" and v["block_n"] == 16
    v = fp8bq.fp8bq_select_variant(4096, 24576, 7168, "fp32", "bf16")
    assert v["from_table"] is False and v["kind"] == "normal" and v["mma_scale"] == 0
    # UE8M0 with whole 4-slab groups: the tensor core applies the scales on
    # wide tiles, not on 16/32-token decode tiles or when K % 512 != 0
    assert fp8bq.fp8bq_select_variant(4096, 24576, 7168, "ue8m0", "bf16")["mma_scale"] == 1
    assert fp8bq.fp8bq_select_variant(128, 24576, 7168, "ue8m0", "bf16")["mma_scale"] == 1
    assert fp8bq.fp8bq_select_variant(8, 24576, 7168, "ue8m0", "bf16")["mma_scale"] == 0
    assert fp8bq.fp8bq_select_variant(4096, 24576, 7296, "ue8m0", "bf16")["mma_scale"] == 0
    # other fmt/out of a tabulated (N,K) also misses
    assert fp8bq.fp8bq_select_variant(1, 4096, 7168, "fp32", "bf16")["from_table"] is False


def test_variant_workspace_bytes():
    v1 = fp8bq.make_variant("swap", 16, 1)
    assert fp8bq.fp8bq_variant_workspace_bytes(8, 7168, 18432, v1) == 0
    v4 = fp8bq.make_variant("swap", 16, 4)
    tiles = 7168 // 128
    assert fp8bq.fp8bq_variant_workspace_bytes(8, 7168, 18432, v4) == \
        65536 + tiles * 4 * 128 * 16 * 4
    # linear: counter prefix + codes + scales (+ partials)
    lin = fp8bq.fp8bq_linear_workspace_bytes(8, 7168, 18432, "ue8m0", "bf16")
    g = fp8bq.fp8bq_gemm_workspace_bytes(8, 7168, 18432, "ue8m0", "bf16")
    codes = (8 * 18432 + 255) // 256 * 256
    scales = (4 * ((144 + 3) // 4) * 8 + 255) // 256 * 256
    assert lin == 65536 + codes + scales + (g - 65536 if g else 0)
    bad = fp8bq.make_variant("swap", 48, 1)
    assert fp8bq.fp8bq_variant_workspace_bytes(8, 7168, 18432, bad) == 0
    # the block-scaled MMA splits K the same way (same partials workspace) ...
    mx4 = fp8bq.make_variant("swap", 16, 4, 0, 1)
    assert fp8bq.fp8bq_variant_workspace_bytes(8, 7168, 18432, mx4) == \
        fp8bq.fp8bq_variant_workspace_bytes(8, 7168, 18432, v4)
    # ... and exists for 128-row tiles only (M = 128 MMAs)
    assert fp8bq.fp8bq_variant_workspace_bytes(
        256, 7168, 18432, fp8bq.make_variant("normal", 128, 2, 0, 1)) > 0
    assert fp8bq.fp8bq_variant_workspace_bytes(
        8, 7168, 18432, fp8bq.make_variant("swap64", 16, 2, 0, 1)) == 0


def call_grouped(E=4, M_max=8, N=128, K=256, ptr=4096, counts=4096, fmt=0, out=0):
    lib = fp8bq.lib()
    p = ctypes.c_void_p(ptr)
    c = None if counts is None else ctypes.c_void_p(counts)
    return lib.fp8bq_grouped_gemm(E, M_max, N, K, c, p, p, p, p, 128, 128, 128, fmt, out, p,
                                  None, 0, None)


def test_grouped_argument_errors_on_host():
    assert call_grouped(E=0) == 1          # no experts
    assert call_grouped(M_max=-4) == 1
    assert call_grouped(M_max=6) == 2      # rows per expert not a multiple of 4
    assert call_grouped(N=192) == 2        # weights not in whole 128-row blocks
    assert call_grouped(K=100) == 2
    assert call_grouped(counts=None) == 1  # counts pointer missing
    assert call_grouped(ptr=4100) == 3
    assert call_grouped(M_max=0) == 0      # empty: no-op
    assert call_grouped(N=0) == 0


def test_grouped_variant_selection_and_workspace():
    # decode-sized experts: swap-AB token tiles from the rows per expert
    v = fp8bq.fp8bq_select_grouped_variant(32, 24, 4096, 7168, "ue8m0", "bf16")
    assert (v["kind"], v["block_n"], v["split"]) == ("swap", 32, 1)
    assert fp8bq.fp8bq_grouped_gemm_workspace_bytes(32, 24, 4096, 7168, "ue8m0", "bf16") == 0
    v = fp8bq.fp8bq_select_grouped_variant(8, 512, 7168, 2048, "fp32", "bf16")
    assert (v["kind"], v["block_n"], v["split"]) == ("normal", 256, 1)
    # few tiles: split K until the GPU's 152 SMs have work (at most 8, at most G)
    v = fp8bq.fp8bq_select_grouped_variant(2, 8, 256, 4096, "fp32", "bf16")
    assert (v["kind"], v["block_n"], v["split"]) == ("swap", 16, 8)
    tiles = 2 * 2 * 1
    assert fp8bq.fp8bq_grouped_gemm_workspace_bytes(2, 8, 256, 4096, "fp32", "bf16") == \
        65536 + tiles * 8 * 128 * 16 * 4
    # stream-K is not offered for grouped problems
    assert fp8bq.fp8bq_grouped_variant_workspace_bytes(
        2, 8, 256, 4096, fp8bq.make_variant("swap", 16, 0)) == 0


def call_rowwise(M=16, N=128, K=256, ptr=4096, sptr=4096, code=0, out=0):
    lib = fp8bq.lib()
    p, s = ctypes.c_void_p(ptr), ctypes.c_void_p(sptr)
    return lib.fp8bq_gemm_rowwise(M, N, K, p, s, p, s, code, out, p, None, 0, None)


def test_rowwise_argument_errors_on_host():
    assert call_rowwise(K=100) == 2        # K % 16
    assert call_rowwise(K=0) == 2
    assert call_rowwise(N=120) == 2        # N % 16
    assert call_rowwise(M=-1) == 1
    assert call_rowwise(code=2) == 1
    assert call_rowwise(out=3) == 1
    assert call_rowwise(ptr=4100) == 3     # codes / out not 16-byte aligned
    assert call_rowwise(sptr=4098) == 3    # scales not 4-byte aligned
    assert call_rowwise(ptr=0) == 1
    assert call_rowwise(M=0) == 0
    lib = fp8bq.lib()
    p = ctypes.c_void_p(4096)
    assert lib.fp8bq_quant_rows(p, 0, 4, 100, 0, p, p, None) == 2
    assert lib.fp8bq_quant_rows(p, 3, 4, 128, 0, p, p, None) == 1      # bad dtype
    assert lib.fp8bq_quant_rows(p, 2, 4, 128, 5, p, p, None) == 1      # bad code
    assert lib.fp8bq_quant_rows(ctypes.c_void_p(4104), 0, 4, 128, 0, p, p, None) == 3
    assert lib.fp8bq_quant_rows(p, 0, 0, 128, 1, p, p, None) == 0
    # the rowwise linear layer takes bf16/fp16 input only
    assert lib.fp8bq_linear_rowwise(p, 2, 4, 128, 128, p, p, 0, 0, p, p, 1 << 20, None) == 4


def test_rowwise_variant_selection_and_workspace():
    # e4m3: promotion-free swap-AB at decode sizes; no block-scaled MMA
    v = fp8bq.fp8bq_select_rowwise_variant(8, 7168, 18432, "e4m3", "bf16")
    assert v["kind"] == "swap" and v["mma_scale"] == 0
    v = fp8bq.fp8bq_select_rowwise_variant(2048, 7168, 18432, "e4m3", "bf16")
    assert v["kind"] == "normal" and v["mma_scale"] == 0
    # int8: the warp-level int8 MMA (swap-AB) up to 64 tokens, the FP8-plane
    # kernel (mma_scale = 1) above
    for M in (1, 48, 64):
        v = fp8bq.fp8bq_select_rowwise_variant(M, 4096, 7168, "int8", "bf16")
        assert v["kind"] == "swap" and v["mma_scale"] == 0
    for M, kind in ((65, "swap"), (2048, "normal")):
        v = fp8bq.fp8bq_select_rowwise_variant(M, 4096, 7168, "int8", "bf16")
        assert v["kind"] == kind and v["mma_scale"] == 1
    # its workspace holds both operands as planes: 2 * Kp bytes per row
    vp = fp8bq.make_variant("normal", 256, 1, 0, 1)
    assert fp8bq.fp8bq_rowwise_variant_workspace_bytes(256, 512, 1040, "int8", vp) == \
        65536 + 256 * 2 * 1152 + 512 * 2 * 1152
    # e4m3 has no block-scaled form
    assert fp8bq.fp8bq_rowwise_variant_workspace_bytes(256, 512, 1024, "e4m3", vp) == 0
    # 8-token tiles: the int8 warp-level kernel only (chosen for M <= 8)
    v8 = fp8bq.make_variant("swap", 8, 2)
    assert fp8bq.fp8bq_rowwise_variant_workspace_bytes(8, 512, 1024, "int8", v8) == \
        65536 + 4 * 2 * 128 * 8 * 4
    assert fp8bq.fp8bq_rowwise_variant_workspace_bytes(8, 512, 1024, "e4m3", v8) == 0
    assert fp8bq.fp8bq_select_rowwise_variant(8, 4096, 7168, "int8", "bf16")["block_n"] == 8
    # a K that is not a multiple of 128 counts its partial last slab
    v4 = fp8bq.make_variant("swap", 16, 4)
    tiles = 7168 // 128
    assert fp8bq.fp8bq_rowwise_variant_workspace_bytes(8, 7168, 1040, "e4m3", v4) == \
        65536 + tiles * 4 * 128 * 16 * 4
    assert fp8bq.fp8bq_rowwise_variant_workspace_bytes(8, 7168, 1040, "int8", v4) == \
        65536 + tiles * 4 * 128 * 16 * 4
    # more splits than the 9 K slabs of K = 1040, and int8 has no normal tiles
    assert fp8bq.fp8bq_rowwise_variant_workspace_bytes(
        8, 7168, 1040, "e4m3", fp8bq.make_variant("swap", 16, 10)) == 0
    assert fp8bq.fp8bq_rowwise_variant_workspace_bytes(
        256, 7168, 1024, "int8", fp8bq.make_variant("normal", 128, 2)) == 0
    # the linear layer's workspace: prefix + codes + scales + parts
    g = fp8bq.fp8bq_rowwise_workspace_bytes(8, 7168, 18432, "int8", "bf16")
    lin = fp8bq.fp8bq_linear_rowwise_workspace_bytes(8, 7168, 18432, "int8", "bf16")
    assert lin == 65536 + 8 * 18432 + 256 + (g - 65536 if g else 0)


def test_int8_block_argument_errors_and_sizes():
    lib = fp8bq.lib()
    p = ctypes.c_void_p(4096)
    g = lambda M=16, N=128, K=256, ptr=4096, grp=128, out=0: lib.fp8bq_gemm_int8_block(  # noqa
        M, N, K, ctypes.c_void_p(ptr), ctypes.c_void_p(ptr), ctypes.c_void_p(ptr),
        ctypes.c_void_p(ptr), grp, 128, 128, out, ctypes.c_void_p(ptr), None, 0, None)
    assert g(K=1040) == 2          # K % 128
    assert g(N=120) == 2           # N % 16
    assert g(grp=64) == 4
    assert g(out=5) == 1
    assert g(ptr=4100) == 3
    assert g(M=0) == 0
    assert lib.fp8bq_quant_act_int8(p, 2, 4, 128, 128, p, p, None) == 4   # fp32 input
    assert lib.fp8bq_quant_act_int8(p, 0, 4, 100, 128, p, p, None) == 2
    assert lib.fp8bq_quant_weight_int8(p, 0, 4, 128, 64, 128, p, p, None) == 4
    # swap-AB only, 8-token tiles allowed; split parts as the FP8 workspace
    v = fp8bq.make_variant("swap", 8, 4)
    tiles = 7168 // 128
    assert lib.fp8bq_int8_block_variant_workspace_bytes(8, 7168, 18432, ctypes.byref(v)) == \
        65536 + tiles * 4 * 128 * 8 * 4
    vn = fp8bq.make_variant("normal", 256, 1)
    assert lib.fp8bq_int8_block_variant_workspace_bytes(256, 512, 1024, ctypes.byref(vn)) == 0
    assert fp8bq.fp8bq_select_int8_block_variant(4, 4096, 7168)["block_n"] == 8
    # above 64 tokens: two e4m3 planes on the promotion kernel (mma_scale = 1)
    v = fp8bq.fp8bq_select_int8_block_variant(2048, 4096, 7168)
    assert v["kind"] == "normal" and v["mma_scale"] == 1
    vp = fp8bq.make_variant("normal", 256, 1, 0, 1)
    assert lib.fp8bq_int8_block_variant_workspace_bytes(256, 512, 1024, ctypes.byref(vp)) == \
        65536 + 256 * 2 * 1024 + 512 * 2 * 1024


def test_header_is_plain_c_and_links(tmp_path):
    """include/fp8bq.h compiles as C11 and a C program links against the
    library and calls it (no C++ or torch types at the boundary)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    src = tmp_path / "t.c"
    src.write_text(
        '#include "fp8bq.h"\n'
        "#include <stdio.h>\n"
        "int main(void) {\n"
        "    fp8bq_variant v;\n"
        "    if (fp8bq_abi_version() != 1) return 1;\n"
        "    /* a host-side argument error, no GPU needed */\n"
        "    if (fp8bq_select_variant(16, 100, 256, FP8BQ_SCALE_FP32, FP8BQ_BF16, &v)\n"
        "        != FP8BQ_ERR_SHAPE) return 2;\n"
        "    printf(\"%s\\n\", fp8bq_status_string(FP8BQ_ERR_SHAPE));\n"
        "    return 0;\n"
        "}\n")
    exe = tmp_path / "t"
    libdir = os.path.dirname(fp8bq.LIB_PATH)
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Werror=implicit-function-declaration",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src),
                        "-L", libdir, "-lfp8bq", "-Wl,-rpath," + libdir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip()


def test_rowwise_table_entries(tmp_path, monkeypatch):
    """rw8 lines of the table give the rowwise e4m3 GEMM its own measured
    shapes (nearest M); int8 and block-path lookups ignore them."""
    t = tmp_path / "rw.tbl"
    t.write_text("7168 18432 rw8 bf16 1 swap 16 2 0 0\n"
                 "7168 18432 rw8 bf16 64 swap 64 2 0 0\n"
                 "7168 18432 ue8m0 bf16 1 swap 16 8 0 1\n")
    monkeypatch.setenv("FP8BQ_TABLE", str(t))
    fp8bq.fp8bq_reload_table()
    try:
        v = fp8bq.fp8bq_select_rowwise_variant(4, 7168, 18432, "e4m3", "bf16")
        assert (v["kind"], v["block_n"], v["split"], v["from_table"]) == ("swap", 16, 2, True)
        v = fp8bq.fp8bq_select_rowwise_variant(50, 7168, 18432, "e4m3", "bf16")
        assert (v["block_n"], v["split"]) == (64, 2)
        # other (N, K) or output dtype: no rw8 entry, the block path's shape / default
        v = fp8bq.fp8bq_select_rowwise_variant(4, 7168, 18432, "e4m3", "fp16")
        assert v["mma_scale"] == 0 and v["from_table"] is False
        # the block path keeps its own entry
        v = fp8bq.fp8bq_select_variant(1, 7168, 18432, "ue8m0", "bf16")
        assert (v["split"], v["mma_scale"]) == (8, 1)
        # int8 never takes e4m3 shapes
        assert fp8bq.fp8bq_select_rowwise_variant(4, 7168, 18432, "int8", "bf16")["block_n"] == 8
    finally:
        monkeypatch.delenv("FP8BQ_TABLE")
        fp8bq.fp8bq_reload_table()


def test_int8_table_entries(tmp_path, monkeypatch):
    """ri8 / bi8 lines give the rowwise INT8 and block INT8 GEMMs measured
    shapes, including the choice between the warp-level kernel (mma_scale 0)
    and the two e4m3 planes (mma_scale 1); an entry the planner rejects falls
    through to the fixed rule."""
    t = tmp_path / "i8.tbl"
    t.write_text("7168 18432 ri8 bf16 32 swap 32 3 0 1\n"
                 "7168 18432 ri8 bf16 96 swap 64 4 0 0\n"
                 "7168 18432 bi8 bf16 16 swap 16 6 0 0\n"
                 "7168 18432 bi8 bf16 2048 swap 128 1 0 1\n"
                 # block_n 8 only exists on the warp-level kernel
                 "2112 7168 bi8 bf16 4 swap 8 1 0 1\n")
    monkeypatch.setenv("FP8BQ_TABLE", str(t))
    fp8bq.fp8bq_reload_table()
    try:
        v = fp8bq.fp8bq_select_rowwise_variant(32, 7168, 18432, "int8", "bf16")
        assert (v["kind"], v["block_n"], v["split"], v["mma_scale"], v["from_table"]) == \
            ("swap", 32, 3, 1, True)
        # nearest M: 100 tokens take the 96-token line (warp-level kernel above
        # the fixed 65-token planes threshold)
        v = fp8bq.fp8bq_select_rowwise_variant(100, 7168, 18432, "int8", "bf16")
        assert (v["block_n"], v["split"], v["mma_scale"]) == (64, 4, 0)
        # e4m3 ignores INT8 lines
        assert fp8bq.fp8bq_select_rowwise_variant(32, 7168, 18432, "e4m3", "bf16")[
            "from_table"] is False
        v = fp8bq.fp8bq_select_int8_block_variant(16, 7168, 18432, "bf16")
        assert (v["block_n"], v["split"], v["mma_scale"], v["from_table"]) == (16, 6, 0, True)
        v = fp8bq.fp8bq_select_int8_block_variant(3000, 7168, 18432, "bf16")
        assert (v["kind"], v["block_n"], v["mma_scale"]) == ("swap", 128, 1)
        # the workspace query follows the table's choice: planes need room
        # for both operands' planes, the warp-level kernel none
        ws_planes = fp8bq.lib().fp8bq_int8_block_workspace_bytes(3000, 7168, 18432,
                                                                 fp8bq._dtype_code("bf16"))
        assert ws_planes >= 2 * 18432 * (3000 + 7168)
        # rejected entry (8-token tile on the planes kernel): the fixed rule
        v = fp8bq.fp8bq_select_int8_block_variant(4, 2112, 7168, "bf16")
        assert (v["block_n"], v["mma_scale"], v["from_table"]) == (8, 0, False)
        # fp16 output: no entry
        assert fp8bq.fp8bq_select_int8_block_variant(16, 7168, 18432, "fp16")[
            "from_table"] is False
    finally:
        monkeypatch.delenv("FP8BQ_TABLE")
        fp8bq.fp8bq_reload_table()


def test_grouped_table_entries(tmp_path, monkeypatch):
    """gue8m0 / gfp32 lines give the grouped (MoE) GEMM measured shapes at the
    nearest rows per expert; the block-scaled MMA is never taken for fp32
    scales, and the plain GEMM ignores grouped lines."""
    t = tmp_path / "g.tbl"
    t.write_text("4096 7168 gue8m0 bf16 16 swap 16 3 0 1\n"
                 "4096 7168 gue8m0 bf16 788 normal 128 1 0 0\n"
                 # stream-K over 32 experts' tiles: more tiles than ticket
                 # counters, so the planner rejects it
                 "4096 7168 gue8m0 bf16 4096 normal 128 0 0 0\n"
                 "4096 7168 gfp32 bf16 16 swap 16 2 0 1\n")
    monkeypatch.setenv("FP8BQ_TABLE", str(t))
    fp8bq.fp8bq_reload_table()
    try:
        v = fp8bq.fp8bq_select_grouped_variant(32, 20, 4096, 7168, "ue8m0", "bf16")
        assert (v["kind"], v["block_n"], v["split"], v["mma_scale"], v["from_table"]) == \
            ("swap", 16, 3, 1, True)
        # the workspace query follows the entry: split parts of 32 experts
        assert fp8bq.fp8bq_grouped_gemm_workspace_bytes(32, 20, 4096, 7168, "ue8m0",
                                                        "bf16") >= 3 * 32 * 20 * 4096 * 4
        v = fp8bq.fp8bq_select_grouped_variant(32, 700, 4096, 7168, "ue8m0", "bf16")
        assert (v["kind"], v["block_n"], v["split"], v["mma_scale"]) == ("normal", 128, 1, 0)
        v = fp8bq.fp8bq_select_grouped_variant(32, 4000, 4096, 7168, "ue8m0", "bf16")
        assert v["from_table"] is False
        # fp32 scales cannot take the block-scaled MMA: the entry falls through
        v = fp8bq.fp8bq_select_grouped_variant(32, 20, 4096, 7168, "fp32", "bf16")
        assert v["from_table"] is False and v["mma_scale"] == 0
        # the plain (non-grouped) GEMM has no entry for this shape
        assert fp8bq.fp8bq_select_variant(16, 4096, 7168, "ue8m0", "bf16")["from_table"] is False
    finally:
        monkeypatch.delenv("FP8BQ_TABLE")
        fp8bq.fp8bq_reload_table()
