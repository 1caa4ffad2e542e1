"""The encode kernel's code decisions, modelled on the CPU.

INT4: k_encode needs rne(r / s_q) (symmetric grid) or floor(r / s_q) (mid-rise grid) with the
IEEE fp32 quotient.  It multiplies r by an approximate reciprocal of s_q instead and
recomputes the quotient with a correctly rounded division only where the product lies
within 2^-17 of a rounding boundary (a half-integer, or an integer for the floor).  The
claim: that gives the IEEE quotient's code for every r.

INT2: the code is decided by comparing r with s_q / 2 (symmetric) or with -s_q, 0, s_q
(mid-rise), all exact in fp32.  The claim: that is the code of the exact quotient r / s_q,
which the fp64 reference takes (an exact half rounds to the even 0).

The model takes the reciprocal as the correctly rounded one moved by up to 4 ulps either
way (the hardware's approximation is within that), computes the product, the boundary test
and the fallback in numpy float32, and compares the codes with those of the IEEE quotient
over every positive finite E4M3 scale, for random r and for r placed within a few ulps of
every boundary."""
import numpy as np
import pytest

import oracle

f32 = np.float32
K_ROUND = f32(1.5 * 2.0 ** 23)
TOL = f32(2.0 ** -17)


def _codes_fast(r, sq, inv, bits, midrise):
    qmax, mid = (1 << (bits - 1)) - 1, 1 << (bits - 1)
    v = (r * inv).astype(f32)
    if midrise:
        fq = np.floor(v)
        close = np.abs((v - np.rint(v)).astype(f32)) < TOL * np.maximum(f32(1), np.abs(v))
        fq = np.where(close, np.floor((r / sq).astype(f32)), fq)
        return np.clip(fq + mid, 0, 2 * mid - 1).astype(np.int64)
    v = np.clip(v, -qmax, qmax).astype(f32)
    tq = (v + K_ROUND).astype(f32)
    d = (v - (tq - K_ROUND).astype(f32)).astype(f32)
    close = np.abs(d) > f32(0.5) - TOL
    exact = np.clip((r / sq).astype(f32), -qmax, qmax).astype(f32)
    tq = np.where(close, (exact + K_ROUND).astype(f32), tq)
    return ((tq - K_ROUND).astype(np.int64) + mid)


def _ulps(x, k):
    """x moved by k fp32 ulps (towards +inf for k > 0)."""
    x = np.asarray(x, dtype=f32)
    for _ in range(abs(k)):
        x = np.nextafter(x, f32(np.inf) if k > 0 else f32(-np.inf)).astype(f32)
    return x


def _codes_ieee(r, sq, bits, midrise):
    qmax, mid = (1 << (bits - 1)) - 1, 1 << (bits - 1)
    q = (r / sq).astype(f32)
    if midrise:
        return np.clip(np.floor(q) + mid, 0, 2 * mid - 1).astype(np.int64)
    return (np.clip(np.rint(q), -qmax, qmax) + mid).astype(np.int64)


@pytest.mark.parametrize("bits", [4])
@pytest.mark.parametrize("midrise", [False, True])
def test_fast_quotient_gives_the_ieee_codes(bits, midrise):
    rng = np.random.default_rng(bits + 2 * midrise)
    sq_all = oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8)).astype(f32)
    top = (1 << (bits - 1)) + 1
    # boundaries: half-integers (symmetric) or integers (floor), inside and just past the grid
    bounds = np.arange(-top, top + 1, dtype=np.float64) + (0.0 if midrise else 0.5)
    for sq in sq_all:
        exact_inv = f32(1.0) / sq
        r_rand = (rng.uniform(-top, top, 400) * sq).astype(f32)
        near = (bounds * float(sq)).astype(f32)
        r_near = np.concatenate([_ulps(near, k) for k in range(-3, 4)])
        r = np.concatenate([r_rand, r_near]).astype(f32)
        want = _codes_ieee(r, sq, bits, midrise)
        for k in range(-4, 5):
            got = _codes_fast(r, sq, _ulps(exact_inv, k), bits, midrise)
            assert np.array_equal(got, want), (bits, midrise, float(sq), k)


def _codes_int2_compare(r, sq, midrise):
    """The kernel's INT2 decision: comparisons with exact multiples of s_q."""
    if midrise:
        return np.where(r >= 0, np.where(r >= sq, 3, 2), np.where(r >= -sq, 1, 0)).astype(np.int64)
    h = f32(0.5) * sq
    return np.where(r > h, 3, np.where(r < -h, 1, 2)).astype(np.int64)


def _codes_exact(r, sq, bits, midrise):
    """Codes of the exact quotient (fp64 is exact enough here: r and s_q have at most 24
    and 4 significant bits, and a boundary is hit only when r is exactly on it)."""
    qmax, mid = (1 << (bits - 1)) - 1, 1 << (bits - 1)
    q = r.astype(np.float64) / float(sq)
    if midrise:
        return np.clip(np.floor(q) + mid, 0, 2 * mid - 1).astype(np.int64)
    return (np.clip(np.rint(q), -qmax, qmax) + mid).astype(np.int64)


@pytest.mark.parametrize("midrise", [False, True])
def test_int2_comparisons_give_the_exact_quotients_codes(midrise):
    rng = np.random.default_rng(11 + midrise)
    sq_all = oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8)).astype(f32)
    bounds = np.array([-1.0, 0.0, 1.0] if midrise else [-1.5, -0.5, 0.5, 1.5])
    n_ieee_differ = 0
    for sq in sq_all:
        r_rand = (rng.uniform(-3, 3, 400) * sq).astype(f32)
        near = (bounds * float(sq)).astype(f32)
        r_near = np.concatenate([_ulps(near, k) for k in range(-3, 4)])
        r = np.concatenate([r_rand, r_near, np.array([0.0, -0.0], dtype=f32)]).astype(f32)
        want = _codes_exact(r, sq, 2, midrise)
        assert np.array_equal(_codes_int2_compare(r, sq, midrise), want), (midrise, float(sq))
        n_ieee_differ += int((_codes_ieee(r, sq, 2, midrise) != want).sum())
    # On the mid-rise grid the IEEE fp32 quotient rounds onto an integer for some r just
    # below it, and the comparisons follow the exact quotient there.  On the symmetric grid
    # the two agree: a quotient by an E4M3 scale (at most 4 significant bits) never rounds
    # onto a half-integer from r off it.
    assert (n_ieee_differ > 0) == midrise
