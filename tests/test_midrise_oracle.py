"""Pins of the oracle's mid-rise scheme (scheme 1), on the CPU.

The reading: one critique of the method says 2-bit codes give "only 4 quantization levels".
The 4-level grid is mid-rise: level u sits at s_q * (u - 2^(b-1) + 1/2), u = 0 .. 2^b - 1,
with s = max|r| / (2^(b-1) - 1/2) stored as E4M3 and u the nearest level (floor(r/s_q) plus
2^(b-1), clamped; a value exactly between two levels takes the upper one).

Each pin ties the oracle to something other than its own encoder: a textbook mid-rise
quantizer written here with numpy, the symmetry of the levels, exact round trips of values
on the grid, the half-step error bound, and the reconstruction identity of the whole path.
"""
import numpy as np
import pytest

import oracle


def _textbook_midrise(R, bits, group):
    """Mid-rise group quantization written out directly (E4M3 scales via the pinned codec)."""
    N, d = R.shape
    mid = 1 << (bits - 1)
    g = R.reshape(N, d // group, group)
    a = np.abs(g).max(axis=2)
    sb = oracle.e4m3_encode(a / (mid - 0.5))
    sq = oracle.e4m3_decode(sb)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(sq > 0, np.floor(g / np.where(sq > 0, sq, 1.0)) + mid, mid)
    u = np.clip(u, 0, 2 * mid - 1).astype(np.int64)
    xhat = sq * (u - mid + 0.5)
    return u.reshape(N, d), sb, xhat.reshape(N, d)


def _unpack(codes, bits):
    per = 8 // bits
    u = np.stack([(codes >> (bits * k)) & ((1 << bits) - 1) for k in range(per)], axis=-1)
    return u.reshape(codes.shape[0], -1).astype(np.int64)


@pytest.mark.parametrize("bits,group", [(2, 16), (2, 32), (2, 64), (4, 16), (4, 64)])
def test_encode_matches_the_textbook_quantizer(bits, group):
    rng = np.random.default_rng(bits * 100 + group)
    R = rng.standard_normal((300, 128)) * rng.choice([0.01, 1.0, 30.0], size=(300, 1))
    R[5] = 0.0  # an all-zero token: s_q = 0
    codes, scales = oracle.encode(R, bits, group, scheme=1)
    u_t, sb_t, xhat_t = _textbook_midrise(R, bits, group)
    np.testing.assert_array_equal(scales, sb_t)
    np.testing.assert_array_equal(_unpack(codes, bits), u_t)
    np.testing.assert_array_equal(oracle.decode_codes(codes, scales, bits, group, scheme=1), xhat_t)


@pytest.mark.parametrize("bits", [2, 4])
def test_levels_are_symmetric_and_there_are_2_to_the_b(bits):
    mid = 1 << (bits - 1)
    # one token whose groups hold every code once (scale byte 0x38 decodes to 1.0)
    u = np.tile(np.arange(2 * mid), 128 // (2 * mid))
    per = 8 // bits
    codes = np.zeros((1, 128 * bits // 8), dtype=np.uint8)
    for k, v in enumerate(u):
        codes[0, k // per] |= np.uint8(v << (bits * (k % per)))
    scales = np.full((1, 128 // 16), 0x38, dtype=np.uint8)
    x = oracle.decode_codes(codes, scales, bits, 16, scheme=1)[0]
    assert oracle.e4m3_decode(np.array([0x38], dtype=np.uint8))[0] == 1.0
    levels = x[: 2 * mid]
    np.testing.assert_array_equal(levels, np.arange(2 * mid) - mid + 0.5)
    np.testing.assert_array_equal(levels, -levels[::-1])
    assert 0.0 not in levels


@pytest.mark.parametrize("bits,group", [(2, 32), (4, 16)])
def test_grid_values_round_trip(bits, group):
    rng = np.random.default_rng(7)
    mid = 1 << (bits - 1)
    N = 64
    sq = 2.0 ** rng.integers(-6, 6, size=(N, 128 // group))  # exact in E4M3
    u = rng.integers(0, 2 * mid, size=(N, 128))
    u[:, ::group] = 2 * mid - 1  # every group reaches its top level, so s = s_q exactly
    R = np.repeat(sq, group, axis=1) * (u - mid + 0.5)
    codes, scales = oracle.encode(R, bits, group, scheme=1)
    np.testing.assert_array_equal(_unpack(codes, bits), u)
    np.testing.assert_array_equal(oracle.decode_codes(codes, scales, bits, group, scheme=1), R)


@pytest.mark.parametrize("bits,group", [(2, 32), (4, 64)])
def test_error_is_at_most_half_a_step(bits, group):
    rng = np.random.default_rng(bits + group)
    mid = 1 << (bits - 1)
    R = rng.standard_normal((400, 128)) * 5.0
    codes, scales = oracle.encode(R, bits, group, scheme=1)
    xhat = oracle.decode_codes(codes, scales, bits, group, scheme=1)
    sq = np.repeat(oracle.e4m3_decode(scales), group, axis=1)
    # half a step inside the grid; past the top level (E4M3 can round s below max|r|/top)
    # the error is the overshoot plus half a step
    bound = 0.5 * sq + np.maximum(0.0, np.abs(R) - (mid - 0.5) * sq)
    assert np.all(np.abs(R - xhat) <= bound * (1 + 1e-12))


def test_whole_path_reconstruction_identity():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((2, 300, 128)) + rng.standard_normal((2, 1, 128)) * 4
    ref = oracle.quantize(X, 8, 2, 2, 32, 3, 5, scheme=1)
    for h in range(2):
        R = oracle.residual(X[h], ref["pi"][h], ref["centroids"][h], 2)
        codes, scales = oracle.encode(R, 2, 32, scheme=1)
        np.testing.assert_array_equal(codes, ref["codes"][h])
        np.testing.assert_array_equal(scales, ref["scales"][h])
        xhat = oracle.dequantize(ref["codes"][h], ref["scales"][h], ref["pi"][h],
                                 ref["centroids"][h], 2, 32, scheme=1)
        want = oracle.decode_codes(codes, scales, 2, 32, scheme=1)
        for t in range(1, -1, -1):
            want = want + ref["centroids"][h][t][ref["pi"][h][t].astype(np.int64)]
        np.testing.assert_array_equal(xhat, want)


def test_scheme_0_is_unchanged_and_the_schemes_differ():
    rng = np.random.default_rng(11)
    R = rng.standard_normal((50, 128))
    c0, s0 = oracle.encode(R, 2, 32)
    c0b, s0b = oracle.encode(R, 2, 32, scheme=0)
    np.testing.assert_array_equal(c0, c0b)
    np.testing.assert_array_equal(s0, s0b)
    c1, s1 = oracle.encode(R, 2, 32, scheme=1)
    assert not np.array_equal(s0, s1)  # a / 1 against a / 1.5


def test_invalid_scheme_is_rejected():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((1, 16, 128)), 4, 1, 2, 32, 1, 0, scheme=2)
