"""The assignment's near-tie margin, modelled on the CPU.

The tensor-core assignment scores s_j = ||c_j||^2 - 2 acc_j with acc_j the fp32-accumulated
product of fp16(r) and the two fp16 planes of c_j (r, c centred on mu), keeps every cluster
whose score is within twice the error bound E of the row's best score, and re-scores those
exactly.  The bound is derived in the header of k_assign.cu:
    E = 2 (1.004 dn cmax + k rn cmax + 2^-20 (rn + dn)) + 1.0625 * 2^-17 cmax^2,
    k = 1.012 * 2^-15, rn = ||r||, dn = ||fp16(r) - r||, cmax = max_j ||c_j||.
This test models those steps in numpy -- fp16 operands, products summed exactly in blocks
of 16 channels (one MMA step), each block added to an fp32 accumulator -- and checks the
claim the choice rests on: the exactly nearest centroid (fp64 distances, ties to the lowest
index) is always among the kept clusters, on random rows, rows with outlier channels and
rows built to sit on near ties."""
import numpy as np
import pytest

f16, f32 = np.float16, np.float32
K_DN, K_RN = f32(1.0 + 1.0 / 256), f32((1.0 + 3.0 / 256) * 2.0 ** -15)


def _kept(R, C):
    """Boolean [N][C]: the clusters the modelled epilogue keeps for each row."""
    mu = C.mean(axis=0, dtype=np.float64).astype(f32)
    r = (R - mu).astype(f32)
    c = (C - mu).astype(f32)
    rh = r.astype(f16).astype(np.float64)
    hi = c.astype(f16)
    lo = (c - hi.astype(f32)).astype(f32).astype(f16)
    cn = (c.astype(np.float64) ** 2).sum(axis=1).astype(f32)
    acc = np.zeros((R.shape[0], C.shape[0]), dtype=f32)
    for plane in (hi, lo):
        p = plane.astype(np.float64)
        for kb in range(0, 128, 16):
            block = rh[:, kb:kb + 16] @ p[:, kb:kb + 16].T   # 16 exact products, summed
            acc = (acc + block.astype(f32)).astype(f32)
    s = (cn[None, :] - f32(2) * acc).astype(f32)
    rn = np.sqrt((r.astype(np.float64) ** 2).sum(axis=1)).astype(f32)
    dn = np.sqrt(((rh - r) ** 2).sum(axis=1)).astype(f32)
    cmax2 = f32(cn.max())
    cmax = f32(np.sqrt(cmax2))
    err = (f32(2) * (K_DN * dn * cmax + K_RN * rn * cmax + f32(2.0 ** -20) * (rn + dn))
           + f32(1.0625 * 2.0 ** -17) * cmax2).astype(f32)
    best = s.min(axis=1)
    lim = (best + (f32(2) * err + f32(1e-30))).astype(f32)
    return s <= lim[:, None]


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
    rng = np.random.default_rng(2)
    R = _outlier_rows(rng, 1500, scale)
    C = R[rng.choice(1500, 256, replace=False)]
    _check(R, C)


def test_rows_built_on_near_ties():
    rng = np.random.default_rng(3)
    C = (rng.standard_normal((64, 128)) * 3).astype(f32)
    a = rng.integers(0, 64, 2000)
    b = (a + rng.integers(1, 64, 2000)) % 64
    mid = 0.5 * (C[a].astype(np.float64) + C[b].astype(np.float64))
    R = (mid + rng.standard_normal((2000, 128)) * 10.0 ** rng.uniform(-7, -2, (2000, 1))).astype(f32)
    multi = _check(R, C)
    assert multi > 0.5    # most of these rows must go to the exact re-scoring


def test_far_from_the_centre():
    # a large common offset: the centring keeps the fp16 operands small
    rng = np.random.default_rng(4)
    R = (rng.standard_normal((1000, 128)) + 500.0).astype(f32)
    C = R[rng.choice(1000, 128, replace=False)]
    _check(R, C)
