"""The cluster sums of a later stage, modelled on the CPU in fp32 (numpy float32, round to
nearest even) and checked against exact rational arithmetic.

From the second stage on, a cluster's members are residuals x - C^(1)[pi^(1)] - ...; the
update kernel forms each one by a TwoSum chain as a running fp32 difference d plus the sum r
of the chain's rounding errors, adds d to a compensated (sum, error) pair and r to the error,
per run of sorted positions inside a 32-position chunk, and the finalize step adds the runs
in chunk order and divides once.  The model replays those steps; the mean must be the fp32
rounding of the exact mean of the exact residuals (what the fp64 oracle stores), except
within 2^-40 of the members' mean size of an fp32 rounding midpoint.  The old way, adding the
fp32-rounded residuals, must miss that on a good share of the same clusters, so the check has
teeth.  The model is not the oracle and the library does not use it."""
from fractions import Fraction

import numpy as np
import pytest

from tests import centroid_model as cm

f32 = np.float32


def two_diff(a, c):
    """a - c as d + err exactly: the kernel's packed form (TwoSum of a and -c)."""
    d = f32(a - c)
    bb = f32(d - a)
    err = f32(f32(a - f32(d - bb)) - f32(c + bb))
    return d, err


def chained(x, cs):
    """The stage input of one channel: x minus the earlier stages' centroid values, as the
    running difference and the sum of the chain's rounding errors."""
    v, r = f32(x), f32(0.0)
    for c in cs:
        v, t = two_diff(v, f32(c))
        r = f32(r + t)
    return v, r


def piece_sum(members, exact_residuals):
    """One run's compensated (sum, error) pair, as the chunk-sum kernel forms it."""
    S, E = f32(0.0), f32(0.0)
    for x, cs in members:
        v, r = chained(x, cs)
        if exact_residuals:
            S, err = cm.two_sum(S, v)
            E = f32(f32(E + err) + r)
        else:  # the fp32-rounded residual fl(v + r)
            S, err = cm.two_sum(S, f32(v + r))
            E = f32(E + err)
    return S, E


def cluster_mean(members, cuts, exact_residuals=True):
    """The finalize step: the runs' pieces added in chunk order (TwoSum of the sums, the
    errors added), then the mean of the compensated total."""
    S, E = f32(0.0), f32(0.0)
    for a, b in zip([0] + cuts, cuts + [len(members)]):
        ps, pe = piece_sum(members[a:b], exact_residuals)
        S, err = cm.two_sum(S, ps)
        E = f32(f32(E + err) + pe)
    return cm.mean_of(S, E, f32(len(members)))


def rne32(q: Fraction) -> np.float32:
    """The fp32 value nearest the rational q, ties to even (no double rounding)."""
    m = float(q)  # nearest double
    f = f32(m)
    if float(f) == m:
        return f
    lo, hi = sorted((f, np.nextafter(f, f32(np.inf) if float(f) < m else f32(-np.inf))))
    mid = (Fraction(float(lo)) + Fraction(float(hi))) / 2
    if q < mid:
        return lo
    if q > mid:
        return hi
    return lo if (lo.view(np.uint32) & 1) == 0 else hi


def near_midpoint(q: Fraction, band: float) -> bool:
    f = rne32(q)
    up = np.nextafter(f, f32(np.inf))
    down = np.nextafter(f, f32(-np.inf))
    mids = [(Fraction(float(f)) + Fraction(float(g))) / 2 for g in (up, down)]
    return any(abs(q - m) <= Fraction(band) for m in mids)


def _clusters(seed, count, stages):
    """Clusters of later-stage residuals built like the synthetic workloads': bf16 token
    values of one channel (ordinary ones about unit size, some outlier channels near 80),
    minus fp32 centroid values of the earlier stages.  A member of a later stage's cluster
    comes from any earlier cluster, so the centroid value it meets is anywhere from near
    zero to near its own value; when it is small against the running difference, that
    difference is not exact in fp32 (the case where rounding the residual loses the most)."""
    import torch
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        n = int(rng.integers(1, 80))
        base = rng.choice([0.0, 1.0, 80.0]) * rng.standard_normal()
        scale = max(1.0, abs(base))
        xs = base + 10.0 ** rng.uniform(-2, 0) * scale * rng.standard_normal(n)
        xs = torch.tensor(xs, dtype=torch.float32).to(torch.bfloat16).float().numpy()
        members = []
        for x in xs:
            cs, rem = [], float(x)
            for _ in range(stages - 1):
                c = f32(rem * rng.uniform(-0.3, 1.0) + 0.1 * abs(rem) * rng.standard_normal())
                cs.append(c)
                rem -= float(c)
            members.append((f32(x), cs))
        cuts = sorted(set(int(c) for c in rng.integers(1, n, size=int(rng.integers(0, 3))))) if n > 1 else []
        out.append((members, cuts))
    return out


def _exact_mean(members):
    tot = Fraction(0)
    for x, cs in members:
        r = Fraction(float(x))
        for c in cs:
            r -= Fraction(float(c))
        tot += r
    return tot / len(members)


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_exact_residual_sums_round_as_the_exact_mean(stages):
    exact_ok = old_wrong = checked = 0
    for members, cuts in _clusters(100 + stages, 400, stages):
        q = _exact_mean(members)
        size = sum(abs(float(_exact_mean([m]))) for m in members) / len(members)
        if near_midpoint(q, 2.0 ** -40 * size):
            continue
        checked += 1
        want = rne32(q)
        got = cluster_mean(members, cuts)
        assert got == want, (stages, float(got), float(want), len(members), cuts)
        exact_ok += 1
        old_wrong += int(cluster_mean(members, cuts, exact_residuals=False) != want)
    assert checked >= 390
    # summing fp32-rounded residuals misses the fp32 rounding of the exact mean often
    assert old_wrong >= 0.1 * checked, old_wrong


def test_first_error_is_exact():
    # one earlier stage: d + err is exactly x - c for bf16 x and fp32 c of similar size
    rng = np.random.default_rng(7)
    for _ in range(2000):
        x = f32(np.float32(rng.standard_normal() * 10.0 ** rng.uniform(-2, 3)))
        c = f32(float(x) * (1 + rng.standard_normal() * 10.0 ** rng.uniform(-6, -1)))
        d, e = two_diff(x, c)
        assert Fraction(float(d)) + Fraction(float(e)) == Fraction(float(x)) - Fraction(float(c))
