"""Pins of the oracle's 16-bit centroid storage (centroid_format 1 = IEEE binary16,
2 = bfloat16), on the CPU.

A 16-bit storage of the centroids takes the residuals against the rounded stored values;
the explainer page's compression ratios count centroids that way, as does the storage
accounting of the presets.  The pins tie the oracle's rounding and its
use to things other than itself:
  * the rounding equals numpy's binary16 cast and torch's bfloat16 cast (both round to
    nearest even), over normal, subnormal, overflowing and tie values;
  * every stored centroid is representable in its format;
  * given the final assignments, each stored centroid is the format's rounding of the exact
    mean of its members, computed here with numpy;
  * the reconstruction identity holds with the rounded centroids;
  * format 0 is the existing fp32 path.
"""
import numpy as np
import pytest
import torch

import oracle


def _edge_values():
    rng = np.random.default_rng(1)
    vals = [rng.standard_normal(4000) * s for s in (1e-7, 1e-5, 1e-3, 1.0, 1e3, 6e4)]
    f16 = np.float16
    # binary16 ties: halfway between neighbours, at normal and subnormal magnitudes
    grid = np.array([1.0, 1.5, 2.0 ** -14, 2.0 ** -20, 65504.0, 1024.0, 2.0 ** -24], dtype=np.float64)
    with np.errstate(over="ignore"):  # the neighbour above 65504 is infinity
        up = np.array([np.nextafter(f16(g), f16(np.inf)) for g in grid], dtype=np.float64)
    ties = (grid + up) / 2
    big = np.array([65504.0, 65519.99, 65520.0, 7e4, -65520.0, 1e300])
    return np.concatenate(vals + [ties, -ties, big, [0.0, -0.0]])


def test_binary16_rounding_matches_numpy():
    x = _edge_values()
    got = oracle.store_centroids(x, 1)
    with np.errstate(over="ignore"):  # past the largest finite value: infinity, as intended
        want = x.astype(np.float16).astype(np.float32)
    np.testing.assert_array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_bfloat16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    # fp32-exact inputs, so torch's cast (which may pass through fp32) is one rounding
    with np.errstate(over="ignore"):  # some of the largest samples overflow to infinity
        x32 = np.concatenate([rng.standard_normal(4000).astype(np.float32) * s for s in
                              (np.float32(1e-38), np.float32(1e-3), np.float32(1.0),
                               np.float32(1e30), np.float32(3e38))])
    # bfloat16 ties: fp32 values exactly halfway between neighbouring bfloat16 values
    base = torch.tensor([1.0, 1.5, 3.0, 2.0 ** -126, 2.0 ** -130], dtype=torch.float32)
    mid = (base.view(torch.int32) + 0x8000).view(torch.float32)
    x32 = np.concatenate([x32, mid.numpy(), -mid.numpy()])
    b = torch.from_numpy(x32).to(torch.bfloat16)
    got = oracle.store_centroids(x32.astype(np.float64), 2)
    np.testing.assert_array_equal(got, b.to(torch.float32).numpy())


@pytest.mark.parametrize("fmt,cast", [(1, np.float16), (2, None)])
def test_stored_centroids_are_rounded_exact_means(fmt, cast):
    rng = np.random.default_rng(5 + fmt)
    X = rng.standard_normal((2, 400, 128)) * 3 + rng.standard_normal((2, 1, 128)) * 10
    C, T = 12, 2
    ref = oracle.quantize(X, C, T, 2, 32, 4, 3, centroid_format=fmt)
    for h in range(2):
        R = X[h].copy()
        for t in range(T):
            cent = ref["centroids"][h][t]
            pi = ref["pi"][h][t].astype(np.int64)
            # representable in the format
            np.testing.assert_array_equal(oracle.store_centroids(cent.astype(np.float64), fmt), cent)
            for j in np.unique(pi):
                m = R[pi == j].mean(axis=0, dtype=np.float64)
                if cast is not None:
                    want = m.astype(cast).astype(np.float32)
                else:
                    want = torch.from_numpy(m).to(torch.bfloat16).to(torch.float32).numpy()
                    # torch rounds fp64 -> bf16 through fp32 (two roundings): allow the one
                    # case that can differ, an fp32 rounding that lands on a bf16 tie
                    diff = want != cent[j]
                    if diff.any():
                        m32 = m.astype(np.float32)
                        assert np.all(np.abs(m[diff] - cent[j][diff]) <=
                                      np.abs(m[diff] - want[diff]) + np.abs(m32[diff] - m[diff]))
                        continue
                np.testing.assert_array_equal(cent[j], want)
            R = R - cent[pi].astype(np.float64)


@pytest.mark.parametrize("fmt", [1, 2])
def test_reconstruction_identity_with_16_bit_centroids(fmt):
    rng = np.random.default_rng(9)
    X = rng.standard_normal((1, 300, 128)) + 5
    ref = oracle.quantize(X, 8, 2, 4, 16, 3, 1, centroid_format=fmt)
    R = oracle.residual(X[0], ref["pi"][0], ref["centroids"][0], 2)
    codes, scales = oracle.encode(R, 4, 16)
    np.testing.assert_array_equal(codes, ref["codes"][0])
    xhat = oracle.dequantize(ref["codes"][0], ref["scales"][0], ref["pi"][0], ref["centroids"][0],
                             4, 16)
    # X = R^(2) + C^(2)[pi] + C^(1)[pi] with the rounded centroids, so the reconstruction
    # error is the codes' error alone (up to fp64 rounding)
    np.testing.assert_allclose(xhat - X[0], oracle.decode_codes(codes, scales, 4, 16) - R,
                               rtol=0, atol=1e-12)


def test_format_0_is_the_fp32_path():
    rng = np.random.default_rng(4)
    X = rng.standard_normal((2, 200, 128))
    a = oracle.quantize(X, 8, 2, 2, 32, 3, 7)
    b = oracle.quantize(X, 8, 2, 2, 32, 3, 7, centroid_format=0)
    for k in ("codes", "scales", "pi", "centroids"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(oracle.store_centroids(X[0, 0], 0), X[0, 0].astype(np.float32))


def test_invalid_format_is_rejected():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((1, 16, 128)), 4, 1, 2, 32, 1, 0, centroid_format=3)
