"""The seeded input generator follows its published definition."""
import numpy as np

import synth


def test_splitmix64_published_sequence():
    # splitmix64 from state 1234567: the first five outputs of the reference C
    # implementation (Vigna, splitmix64.c), as used by common test suites.
    state = 1234567
    got = []
    for _ in range(5):
        state = (state + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        got.append(int(synth._mix(np.array([state], dtype=np.uint64))[0]))
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_streams_are_slab_consistent_and_distinct():
    full = synth.normal(0, 1, 0, 1000)
    np.testing.assert_array_equal(full[337:600], synth.normal(0, 1, 337, 263))
    assert not np.array_equal(full[:100], synth.normal(0, 2, 0, 100))
    x = synth.activations_bf16(0, 8, 256, 4, 20.0)
    np.testing.assert_array_equal(x[3:6], synth.activations_bf16(0, 3, 256, 4, 20.0, row0=3))


def test_normal_moments_and_outliers():
    v = synth.normal(0, 0, 0, 1 << 20)
    assert abs(v.mean()) < 5e-3 and abs(v.std() - 1) < 5e-3
    cols = synth.outlier_columns(0, 4096, 41)
    assert len(np.unique(cols)) == 41 and cols.min() >= 0 and cols.max() < 4096
    ids = synth.token_ids(0, 8192, 248000)
    assert ids.min() >= 0 and ids.max() < 248000
