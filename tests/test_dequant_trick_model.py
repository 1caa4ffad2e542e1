"""The fused dequant's level trick, modelled on the CPU over every case.

The kernel turns a packed code into its level without an integer-to-float conversion: the
code u (field e of a 16-bit word, shifted left by sh = 1 on the mid-rise grid) is masked
into the mantissa of the float 2^23, one fp32 subtraction of 2^23 + (MID * 2^sh - sh) * 2^(b e)
leaves (2^sh (u - MID) + sh) * 2^(b e) exactly, and multiplying by s_q * 2^-(b e + sh) gives
s_q * (u - MID) (symmetric grid) or s_q * (u - MID + 1/2) (mid-rise), exactly.

This test restates those steps with numpy uint32 / float32 operations and checks them
against the level computed in fp64, for both bit widths, both grids, every field of the
word, every code (with random neighbouring codes in the word) and every finite E4M3 scale."""
import numpy as np
import pytest

import oracle

f32 = np.float32


def _float_bits(u32):
    return np.asarray(u32, dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("sh", [0, 1])
def test_level_trick_is_exact(bits, sh):
    mid = 1 << (bits - 1)
    per16 = 16 // bits
    sq = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float32)  # finite, >= 0
    sq = np.concatenate([sq, -sq[1:]])
    rng = np.random.default_rng(bits * 2 + sh)
    for e in range(per16):
        se = (sq * _float_bits((127 - bits * e - sh) << 23)).astype(f32)   # s_q * 2^-(b e + sh)
        ke = f32(_float_bits(0x4B000000)) + f32(((mid << sh) - sh) << (bits * e))
        for u in range(1 << bits):
            others = rng.integers(0, 1 << 16, size=sq.size, dtype=np.uint32)
            keep = np.uint32(0xFFFF & ~(((1 << bits) - 1) << (bits * e)))
            word = (others & keep) | np.uint32(u << (bits * e))
            word = (word << sh).astype(np.uint32)
            m = (word & np.uint32(((1 << bits) - 1) << (bits * e + sh))) | np.uint32(0x4B000000)
            y = (_float_bits(m) - ke).astype(f32)
            assert np.all(y == f32((2 ** sh * (u - mid) + sh) * 2.0 ** (bits * e)))
            x = (se * y).astype(f32)
            level = (u - mid) + 0.5 * sh
            np.testing.assert_array_equal(x.astype(np.float64), sq.astype(np.float64) * level)
