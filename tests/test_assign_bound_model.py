"""The assignment's near-tie margin, modelled on the CPU.

With a = r - mu and c_j = C_j - mu (fp32), the tensor cores accumulate in fp32 the score
t_j = -||c_j||^2 / 2 + fp16(a).fp16(c_j): the offset first (an exact three-part tf32 split of
the fp32 value), then eight MMA steps of 16 channels.  The epilogue keeps every cluster whose
score is within twice the error bound E of the row's best score, and those are re-scored
exactly.  The bound is derived in the header of k_assign.cu:
    E = 1.01 dn (cmax + dcmax) + 1.01 rn dcmax + 2^-15 ((rn + dn)(cmax + dcmax) + cmax^2)
        + 2^-20 (rn + dn),
    rn = ||a||, dn = ||fp16(a) - a||, cmax = max_j ||c_j||, dcmax = max_j ||fp16(c_j) - c_j||.
This test models those steps in numpy -- fp16 operands, products summed exactly in blocks of
16 channels (one MMA step), each block rounded to fp32 and added to the fp32 accumulator --
and checks the claim the choice rests on: the exactly nearest centroid (fp64 distances, ties
to the lowest index) is always among the kept clusters, on random rows, rows with outlier
channels, rows far from the centre and rows built to sit on near ties.  A margin ten times
narrower loses the nearest centroid on the near-tie rows, so the bound is not loose by that
much."""
import numpy as np
import pytest

f16, f32 = np.float16, np.float32
K_DN = f32(1.0 + 3.0 / 256)   # 1.01 as the kernel's constant 0x1.03p0
K_ACC = f32(2.0 ** -15)


def _kept(R, C, narrow=1.0):
    """Boolean [N][C]: the clusters the modelled epilogue keeps for each row."""
    mu = C.mean(axis=0, dtype=np.float64).astype(f32)
    a = (R - mu).astype(f32)
    c = (C - mu).astype(f32)
    ah = a.astype(f16).astype(np.float64)
    ch = c.astype(f16).astype(np.float64)
    cn = (c.astype(np.float64) ** 2).sum(axis=1).astype(f32)      # fp32 sum of squares
    acc = np.repeat((f32(-0.5) * cn)[None, :], R.shape[0], axis=0).astype(f32)
    for kb in range(0, 128, 16):
        block = ah[:, kb:kb + 16] @ ch[:, kb:kb + 16].T            # 16 exact products, summed
        acc = (acc + block.astype(f32)).astype(f32)
    rn = np.sqrt((a.astype(np.float64) ** 2).sum(axis=1)).astype(f32)
    dn = np.sqrt(((ah - a) ** 2).sum(axis=1)).astype(f32)
    dc = np.sqrt(((ch - c) ** 2).sum(axis=1)).astype(f32)
    cmax2 = f32(cn.max())
    cmax = f32(np.sqrt(cmax2) * 1.000001)
    dcmax = f32(dc.max())
    cm1 = f32(cmax + dcmax)
    err = (K_DN * dn * cm1 + K_DN * rn * dcmax + K_ACC * ((rn + dn) * cm1 + cmax2)
           + f32(2.0 ** -20) * (rn + dn)).astype(f32)
    best = acc.max(axis=1)
    lim = (best - (f32(2) * err * f32(narrow) + f32(1e-30))).astype(f32)
    return acc >= lim[:, None]


def _nearest(R, C):
    D = ((R.astype(np.float64)[:, None, :] - C.astype(np.float64)[None, :, :]) ** 2).sum(axis=2)
    return D.argmin(axis=1)


def _check(R, C):
    kept = _kept(R, C)
    j = _nearest(R, C)
    assert kept[np.arange(R.shape[0]), j].all()
    return float((kept.sum(axis=1) > 1).mean())


def _outlier_rows(rng, n, scale):
    X = rng.standard_normal((n, 128)) * scale
    X[:, :4] += rng.choice([-1, 1], 4) * rng.uniform(60, 90, 4) * scale
    return X.astype(f32)


def test_random_rows():
    rng = np.random.default_rng(1)
    R = rng.standard_normal((1500, 128)).astype(f32)
    C = R[rng.choice(1500, 256, replace=False)] + rng.standard_normal((256, 128)).astype(f32) * 0.1
    multi = _check(R, C.astype(f32))
    assert multi < 0.05   # near ties are rare on random rows


@pytest.mark.parametrize("scale", [1.0, 10.0])
def test_rows_with_outlier_channels(scale):
    # the value tensors' case: outlier channels of 600-900 give ||c||^2 far beyond the fp16
    # range, which the tf32 offset carries
    rng = np.random.default_rng(2)
    R = _outlier_rows(rng, 1500, scale)
    C = R[rng.choice(1500, 256, replace=False)]
    _check(R, C)


def _near_tie_rows(seed):
    rng = np.random.default_rng(seed)
    C = (rng.standard_normal((64, 128)) * 3).astype(f32)
    a = rng.integers(0, 64, 2000)
    b = (a + rng.integers(1, 64, 2000)) % 64
    mid = 0.5 * (C[a].astype(np.float64) + C[b].astype(np.float64))
    R = (mid + rng.standard_normal((2000, 128)) * 10.0 ** rng.uniform(-7, -2, (2000, 1))).astype(f32)
    return R, C


def test_rows_built_on_near_ties():
    R, C = _near_tie_rows(3)
    multi = _check(R, C)
    assert multi > 0.5    # most of these rows must go to the exact re-scoring


def test_a_narrower_margin_loses_the_nearest_centroid():
    R, C = _near_tie_rows(3)
    kept = _kept(R, C, narrow=0.1)
    j = _nearest(R, C)
    assert not kept[np.arange(R.shape[0]), j].all()


def test_far_from_the_centre():
    # a large common offset: the centring keeps the fp16 operands small
    rng = np.random.default_rng(4)
    R = (rng.standard_normal((1000, 128)) + 500.0).astype(f32)
    C = R[rng.choice(1000, 128, replace=False)]
    _check(R, C)


def test_offset_split_is_exact():
    # the kernel's three tf32 parts of -||c||^2 / 2 add back to the fp32 value exactly, and
    # each part has at most 11 significant bits
    rng = np.random.default_rng(5)
    v = (-(rng.standard_normal(20000) ** 2) * 10.0 ** rng.uniform(-6, 12, 20000)).astype(f32)

    def tf32(x):
        b = (np.asarray(x, f32).view(np.uint32).astype(np.uint64) + 0x1000) & 0xFFFFE000
        return b.astype(np.uint32).view(f32)

    h = tf32(v)
    r = (v - h).astype(f32)
    m = tf32(r)
    low = (r - m).astype(f32)
    assert np.all(h.astype(np.float64) + m.astype(np.float64) + low.astype(np.float64) == v)
    for part in (h, m, low):
        assert np.all((part.view(np.uint32) & 0x1FFF) == 0)
