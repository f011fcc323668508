"""Host checks of the seeded input generators (no GPU needed)."""

import numpy as np

import workloads


def test_moe_routing_counts():
    c = workloads.moe_routing(0, 1000, 16, 4, 1.1)
    assert c.sum() == 4000 and len(c) == 16
    assert c[0] > c[-1]        # skewed towards low ranks
    assert c.max() <= 1000     # an expert takes a token at most once
    assert np.array_equal(c, workloads.moe_routing(0, 1000, 16, 4, 1.1))   # seeded


def test_bf16_rounding_is_round_to_nearest_even():
    a = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5], dtype=np.float32)
    r = workloads.bf16_round(a)
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == 1.0 + 2 ** -7 and r[3] == -2.5


def test_activation_has_planted_mean():
    x = workloads.activation(workloads.rng(0), 4096, 64, spike=50.0)
    mu = x.astype(np.float64).mean(axis=0)
    assert np.std(mu) > 4.0          # |mu_j| ~ 8 N(0, 1), dominating the N(0, 1) noise
