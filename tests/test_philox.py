"""Pins of the Philox4x32-10 generator to the published known-answer vectors."""
import os

import numpy as np

from workloads.philox import philox4x32_10, philox_uniforms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            w = [int(x, 16) for x in line.split()]
            yield w[:4], w[4:6], w[6:10]


def test_known_answer_vectors():
    cases = list(_kat())
    assert len(cases) == 3
    for ctr, key, want in cases:
        assert [int(x) for x in philox4x32_10(ctr, key)] == want


def test_uniforms_are_24_bit_and_in_range():
    u = philox_uniforms(100_000, seed=0)
    assert u.dtype == np.float32
    assert (u >= 0).all() and (u < 1).all()
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))
    assert abs(u.mean() - 0.5) < 0.005
    # counter-based: any slice equals the matching window of a longer draw
    np.testing.assert_array_equal(philox_uniforms(10, seed=0, offset=500), u[500:510])
    assert not np.array_equal(philox_uniforms(10, seed=1), u[:10])
