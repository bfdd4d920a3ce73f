"""The seeded input generators' own properties (no method arithmetic): the
benchmark-sized row-blocked draws give a row the same values whatever the
number of rows drawn (so a test can take the first M rows of one draw as the
M-row input), and the parallel bf16 conversion gives the serial one's bits."""
import numpy as np

from block_scaled_fp8_group_gb300 import synth


def test_blocked_rows_depend_only_on_seed_and_row():
    a = synth.normal_blocked((2500, 96), seed=3)
    b = synth.normal_blocked((1100, 96), seed=3)
    assert np.array_equal(a[:1100], b)
    assert not np.array_equal(a[:1024], synth.normal_blocked((1024, 96), seed=4))
    x = synth.act_full_grid_blocked(1500, 512)
    assert np.array_equal(x[:300], synth.act_full_grid_blocked(300, 512))


def test_parallel_bf16_conversion_matches_serial():
    x = synth.normal_blocked((3000, 64), seed=5) * np.float32(37.0)
    assert np.array_equal(synth.f32_to_bf16_bits_par(x, block_rows=256),
                          synth.f32_to_bf16_bits(x))


def test_blocked_distributions():
    w = synth.bf16_bits_to_f32(synth.weight_bf16_blocked(2048, 256)).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.001 and abs(w.mean()) < 0.001
    t = synth.bf16_bits_to_f32(synth.act_prefill_blocked(1200, 256)).astype(np.float64)
    assert abs(np.sqrt(np.mean(t * t)) - 1.0) < 0.01
