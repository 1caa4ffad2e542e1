"""The exact re-scoring's fp32-or-fp64 decision, modelled on the CPU.

k_refine orders a near-tie row's candidate clusters by fp32 distances from the fp32 stage
input and settles close calls in fp64 on the stage input rebuilt in fp64.  From the second
stage on, the fp32 stage input is itself rounded (at most 2^-24 |x_k| per channel), which
can reorder two distances whose relative gap is wider than the fp32 arithmetic alone
explains, when the row is much larger than its distances to the candidates.  The margin
for the fp64 decision therefore adds 2^-22 ||x|| sqrt(D_2) to 2^-18 D_2.

The model builds such rows on purpose (the second centroid displaced along the pattern of
the input's rounding, the exact gap between 2^-18 and 2^-12 of the distance), computes the
fp32 distances as the kernel does (one half-warp per row: a fused chain of 8 channels per
lane, then a butterfly sum over the 16 lanes) and checks that every wrongly ordered pair is
sent to fp64 -- which the margin without the input term would not do."""
import numpy as np

f32 = np.float32


def _d32(x32, c):
    d = (x32 - c).astype(f32).reshape(16, 8).astype(np.float64)
    lane = (d[:, 0] * d[:, 0]).astype(f32)
    for k in range(1, 8):
        lane = (d[:, k] * d[:, k] + lane.astype(np.float64)).astype(f32)   # fma: exact product
    for o in (8, 4, 2, 1):
        lane = (lane + lane[np.arange(16) ^ o]).astype(f32)
    assert np.all(lane == lane[0])   # the butterfly leaves every lane with the same sum
    return lane[0]


def test_input_rounding_term_sends_every_misordered_pair_to_fp64():
    rng = np.random.default_rng(1)
    wrong = escaped_old = escaped_new = 0
    for _ in range(3000):
        x = rng.standard_normal(128) * 10.0 ** rng.uniform(1, 3)      # exact stage input
        x32 = x.astype(f32)
        delta = x32.astype(np.float64) - x
        sgn = np.where(delta >= 0, 1.0, -1.0)
        dist = 10.0 ** rng.uniform(-2, 0)
        gap = 2.0 ** rng.uniform(-18, -12) * dist ** 2
        v = sgn * (4 * gap / (2 * np.abs(delta).sum()))
        nv = np.linalg.norm(v)
        if not nv < dist:
            continue
        perp = rng.standard_normal(128)
        perp -= perp @ v / nv ** 2 * v
        perp /= np.linalg.norm(perp)
        alpha = nv / 2 - gap / (2 * nv)
        w = perp * np.sqrt(dist ** 2 - alpha ** 2) + alpha * v / nv
        c1 = (x - w).astype(f32)
        c2 = (c1.astype(np.float64) + v).astype(f32)
        D1 = ((x - c1) ** 2).sum()
        D2 = ((x - c2) ** 2).sum()
        if D1 == D2:
            continue
        a, b = _d32(x32, c1), _d32(x32, c2)
        if (a <= b) == (D1 < D2):
            continue
        wrong += 1
        best, second = min(a, b), max(a, b)
        old = second - best <= f32(2.0 ** -18) * second
        xn = f32(np.sqrt((x32.astype(np.float64) ** 2).sum()))
        new = second - best <= f32(2.0 ** -18) * second + f32(1.0625 * 2.0 ** -22) * xn * f32(np.sqrt(second))
        escaped_old += int(not old)
        escaped_new += int(not new)
    assert wrong > 100 and escaped_old > 50
    assert escaped_new == 0
