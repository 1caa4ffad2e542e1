"""The 16-bit centroid rounding rule, modelled on the CPU (tests/centroid_model.py) and
checked against the oracle at constructed ties.

A cluster whose exact mean lies a third of an fp32 ulp above (or below) the midpoint of two
binary16 / bfloat16 values has an fp32 mean exactly on that midpoint.  Rounding the fp32
mean alone then takes the even neighbour, half the time the wrong one; the rule uses the
sign of what the fp32 mean leaves out and must give the oracle's rounding of the exact mean
in every case, and round to even on an exact tie."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import centroid_model as cm

f32 = np.float32


def _midpoints(fmt, count, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        v = f32(rng.choice([-1.0, 1.0]) * 2.0 ** rng.uniform(-10, 12))
        lo, hi, _ = cm._neighbours(v, fmt)
        if lo == hi:
            continue
        mid = f32(0.5 * (lo + hi))
        if float(mid) == 0.5 * (lo + hi):
            out.append(mid)
    return out


def _exact_mean(xs):
    return float(sum(Fraction(float(x)) for x in xs) / len(xs))


@pytest.mark.parametrize("fmt", [1, 2])
def test_rule_matches_the_oracle_at_constructed_ties(fmt):
    naive_wrong = 0
    for k, m in enumerate(_midpoints(fmt, 300, fmt)):
        u = np.spacing(np.abs(m))  # one fp32 ulp at m
        for offset in (+1, -1, 0):
            # three members: the exact mean is m + offset * u / 3
            xs = [f32(m + offset * u), m, m]
            exact = _exact_mean(xs)
            want = oracle.store_centroids(np.array([exact]), fmt)[0]
            got = cm.stored_mean(xs, fmt)
            assert got == want, (fmt, float(m), offset, float(got), float(want))
            assert cm.mean_of(*cm.compensated_sum(xs), f32(3)) == m  # the fp32 mean is the tie
            naive = cm.store_value(m, f32(0.0), fmt)
            naive_wrong += int(naive != want)
    # rounding the fp32 mean alone is wrong on about half of the off-centre cases
    assert naive_wrong > 100


@pytest.mark.parametrize("fmt", [1, 2])
def test_rule_matches_the_oracle_on_random_clusters(fmt):
    rng = np.random.default_rng(10 + fmt)
    for _ in range(400):
        n = int(rng.integers(1, 40))
        xs = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 3)).astype(f32)
        want = oracle.store_centroids(np.array([_exact_mean(xs)]), fmt)[0]
        assert cm.stored_mean(xs, fmt) == want
