"""The e4m3 tables of the INT8 plane split (quant.cu, int8_planes_kernel):
every int8 code q must split into planes whose e4m3 values are 16*(q >> 4)
and q & 15 (so they sum to q), decoded with the oracle's own e4m3 decoder.
The kernel's byte-permute lookup is replayed here on the CPU with the
constants read from the kernel source, so the test checks what the GPU uses."""
import os
import re

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def kernel_tables():
    src = open(os.path.join(ROOT, "block_scaled_fp8_group_gb300", "csrc", "quant.cu")).read()
    calls = re.findall(r"nibble_lut\(([^;]*)\);", src)
    tabs = []
    for c in calls:
        words = re.findall(r"0x([0-9A-Fa-f]{8})u", c)
        if len(words) >= 4:  # the nibble mask, then the table's four words
            tabs.append([int(w, 16) for w in words[-4:]])
    assert len(tabs) == 2, "expected the l table and the 16h table"
    return tabs  # [l table, 16h table], in the order of the kernel's calls


def byte_perm(x, y, s):
    """__byte_perm with selector nibbles of at most 7 (no sign replication)."""
    b = [(x >> (8 * i)) & 0xFF for i in range(4)] + [(y >> (8 * i)) & 0xFF for i in range(4)]
    return sum(b[(s >> (4 * n)) & 7] << (8 * n) for n in range(4))


def nibble_lut(n, t):
    sel = (n & 0x7) | ((n >> 4) & 0x70) | ((n >> 8) & 0x700) | ((n >> 12) & 0x7000)
    lo, hi = byte_perm(t[0], t[1], sel), byte_perm(t[2], t[3], sel)
    m = ((n >> 3) & 0x01010101) * 0xFF
    return (lo & ~m & 0xFFFFFFFF) | (hi & m)


def test_every_code_splits_exactly():
    lt, ht = kernel_tables()
    dec = oracle.e4m3_decode_all()
    for q in range(-128, 128):
        w = (q & 0xFF) * 0x01010101  # the code in all four byte lanes
        lo = nibble_lut(w & 0x0F0F0F0F, lt)
        hi = nibble_lut((w >> 4) & 0x0F0F0F0F, ht)
        for j in range(4):  # every lane gives the same codes
            lj, hj = (lo >> (8 * j)) & 0xFF, (hi >> (8 * j)) & 0xFF
            assert dec[lj] == (q & 15), (q, j)
            assert dec[hj] == 16 * (q >> 4), (q, j)
            assert dec[hj] + dec[lj] == q


def test_mixed_lanes():
    lt, ht = kernel_tables()
    dec = oracle.e4m3_decode_all()
    for codes in ((-128, 127, -1, 0), (15, 16, -16, -17), (85, -86, 7, -8)):
        w = sum((c & 0xFF) << (8 * j) for j, c in enumerate(codes))
        lo = nibble_lut(w & 0x0F0F0F0F, lt)
        hi = nibble_lut((w >> 4) & 0x0F0F0F0F, ht)
        for j, c in enumerate(codes):
            assert dec[(hi >> (8 * j)) & 0xFF] + dec[(lo >> (8 * j)) & 0xFF] == c
