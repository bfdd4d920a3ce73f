"""The bench's per-GEMM metric formulas against the numbers the pages print:
every row of the DeepGEMM H100 table ("vLLM DeepGEMM FP8 Block GEMM 基准测试"
§3.2, formulas of §4.3) must be reproduced by TFLOPS = gemm_flops / t and
GB/s = pages_gbs_bytes / t from its printed time, within the rounding of the
printed figures (time to 0.1 us, TFLOPS and GB/s to 0.1).  A dropped term
(say 2*m*n), a factor of two or a transposed operand count fails rows."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

TABLE = os.path.join(ROOT, "tests", "golden", "deepgemm_h100_table.txt")


def rows():
    out = []
    for line in open(TABLE, encoding="utf-8"):
        body = line.split("#")[0].split()
        if body:
            m, n, k = (int(x) for x in body[:3])
            t, tf, gbs = (float(x) for x in body[3:])
            out.append((m, n, k, t, tf, gbs))
    return out


def bracket(numerator, t_us, scale):
    """The values a figure can take when the time was rounded to 0.1 us."""
    lo = numerator / ((t_us + 0.05) * 1e-6) / scale
    hi = numerator / ((t_us - 0.05) * 1e-6) / scale
    return lo - 0.05, hi + 0.05


@pytest.mark.parametrize("m,n,k,t,tf,gbs", rows())
def test_pages_table_row(m, n, k, t, tf, gbs):
    lo, hi = bracket(bench.gemm_flops(m, n, k), t, 1e12)
    assert lo <= tf <= hi, (lo, tf, hi)
    lo, hi = bracket(bench.pages_gbs_bytes(m, n, k), t, 1e9)
    assert lo <= gbs <= hi, (lo, gbs, hi)


def test_table_complete():
    assert len(rows()) == 16
