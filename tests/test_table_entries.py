"""Every entry of the committed GB300 table is one the kernels have: the
planner accepts it for its shape and format, and the lookup at its own M
returns it unchanged.  A kernel change that drops a shape, or a hand edit
that names one, fails here instead of silently falling back to the default
rule on the GPU (host-only; launches nothing)."""
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "block_scaled_fp8_group_gb300", "tables", "NVIDIA_GB300.tbl")
E_TUNED = 32  # grouped entries were measured over the MoE workload's 32 local experts


def entries():
    out = []
    for line in open(TABLE):
        body = line.split("#")[0].split()
        if body:
            out.append(body)
    return out


@pytest.fixture(scope="module")
def fp8bq():
    from block_scaled_fp8_group_gb300 import build
    build.build()
    from block_scaled_fp8_group_gb300 import fp8bq as m
    old = os.environ.get("FP8BQ_TABLE")
    os.environ["FP8BQ_TABLE"] = TABLE
    m.fp8bq_reload_table()
    yield m
    if old is None:
        del os.environ["FP8BQ_TABLE"]
    else:
        os.environ["FP8BQ_TABLE"] = old
    m.fp8bq_reload_table()


def test_every_line_parses():
    rows = entries()
    assert len(rows) > 300
    for body in rows:
        assert len(body) == 10, body
        assert body[2] in ("fp32", "ue8m0", "rw8", "ri8", "bi8", "gfp32", "gue8m0"), body
        assert body[3] in ("bf16", "fp16", "fp32") and body[5] in ("normal", "swap", "swap64")


def test_every_entry_is_supported_and_found(fp8bq):
    checked = 0
    for body in entries():
        N, K = int(body[0]), int(body[1])
        fmt, out, M = body[2], body[3], int(body[4])
        want = (body[5], int(body[6]), int(body[7]), int(body[9]))
        if fmt in ("fp32", "ue8m0"):
            v = fp8bq.make_variant(body[5], int(body[6]), int(body[7]), int(body[8]), int(body[9]))
            assert fp8bq.fp8bq_variant_supported(M, N, K, fmt, v), body
            got = fp8bq.fp8bq_select_variant(M, N, K, fmt, out)
        elif fmt in ("rw8", "ri8"):
            got = fp8bq.fp8bq_select_rowwise_variant(M, N, K, "e4m3" if fmt == "rw8" else "int8",
                                                     out)
        elif fmt == "bi8":
            got = fp8bq.fp8bq_select_int8_block_variant(M, N, K, out)
        else:
            got = fp8bq.fp8bq_select_grouped_variant(E_TUNED, M, N, K, fmt[1:], out)
        assert got["from_table"] is True, body
        assert (got["kind"], got["block_n"], got["split"], got["mma_scale"]) == want, body
        checked += 1
    assert checked == len(entries())


def test_variant_supported_rejects(fp8bq):
    """The check itself: shapes the kernels lack are refused."""
    mx = fp8bq.make_variant("swap", 16, 1, 0, 1)
    assert fp8bq.fp8bq_variant_supported(8, 7168, 18432, "ue8m0", mx)
    assert not fp8bq.fp8bq_variant_supported(8, 7168, 18432, "fp32", mx)   # fp32 scales
    assert not fp8bq.fp8bq_variant_supported(8, 7168, 1152, "ue8m0", mx)   # K % 512 != 0
    assert not fp8bq.fp8bq_variant_supported(8, 7168, 18432, "fp32",
                                             fp8bq.make_variant("swap", 24, 1))  # token tile
    assert not fp8bq.fp8bq_variant_supported(8, 7168, 18432, "fp32",
                                             fp8bq.make_variant("normal", 64, 1))
