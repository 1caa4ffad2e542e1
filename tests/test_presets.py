"""The presets and the storage accounting, on the CPU.

Pins:
  * The pages print about 6.4x compression for the INT2 baselines at block size 16 with
    per-group scales.  That is plain group quantization (no stages), where the accounting
    is 16 / (2 + 8/16) = 6.4 exactly.
  * They print about 6.94x for QVG (one stage, B = 64) and about 5.0x for QVG-Pro (four
    stages, B = 16) on LongCat-Video at INT2.  With 16-bit centroids and a cache of the
    pages' size (about 35 000 tokens per tensor) the accounting gives both within a few
    percent.
  * The quantized values take most of the storage (the pages say 65 % or more; that holds
    for QVG, and for QVG-Pro the codes remain the largest part).
  * The accounting equals the bytes of the buffers the library actually allocates.
"""
import pytest

from video_kv_cache_gb300 import api
from video_kv_cache_gb300.presets import PRESETS, cache_bytes, storage_bits


def test_rtn_baseline_ratio_is_the_printed_6_4():
    r = storage_bits(bits=2, group=16, T=0, C=0, N=1000)
    assert r["compression_ratio"] == pytest.approx(6.4, abs=1e-12)


@pytest.mark.parametrize("name,printed", [("qvg", 6.94), ("qvg_pro", 5.0)])
def test_preset_ratios_match_the_printed_ones(name, printed):
    p = PRESETS[name]
    r = storage_bits(p.bits, p.group, p.T, p.C, N=35000, centroid_bits=16)
    assert abs(r["compression_ratio"] - printed) / printed < 0.03, r


def test_presets_are_the_pages_settings():
    assert (PRESETS["qvg"].T, PRESETS["qvg"].group) == (1, 64)
    assert (PRESETS["qvg_pro"].T, PRESETS["qvg_pro"].group) == (4, 16)
    for p in PRESETS.values():
        assert p.bits == 2 and p.C == 256


def test_codes_dominate_the_storage():
    # the pages' ">= 65 %" holds for QVG at either centroid width; QVG-Pro's four stages of
    # metadata bring the codes to about 60 % at a cache of this size, still the largest part
    for cb in (16, 32):
        p = PRESETS["qvg"]
        r = storage_bits(p.bits, p.group, p.T, p.C, N=32760, centroid_bits=cb)
        assert r["codes_share"] >= 0.65, (cb, r)
        p = PRESETS["qvg_pro"]
        r = storage_bits(p.bits, p.group, p.T, p.C, N=32760, centroid_bits=cb)
        parts = r["bits_per_element"]
        assert parts["codes"] == max(parts.values()), (cb, r)


def test_more_stages_or_smaller_groups_cost_more_bits():
    base = storage_bits(2, 64, 1, 256, 32760)["total_bits_per_element"]
    assert storage_bits(2, 16, 1, 256, 32760)["total_bits_per_element"] > base
    assert storage_bits(2, 64, 4, 256, 32760)["total_bits_per_element"] > base


@pytest.mark.parametrize("name", sorted(PRESETS))
@pytest.mark.parametrize("N", [1000, 32760])
def test_accounting_equals_allocated_bytes(name, N):
    p = PRESETS[name]
    H = 3
    ckv = api.allocate(H, N, p.C, p.T, p.bits, p.group, device="cpu")
    r = storage_bits(p.bits, p.group, p.T, p.C, N, centroid_bits=32)
    want_bits = r["total_bits_per_element"] * H * N * 128
    assert cache_bytes(ckv, N) * 8 == pytest.approx(want_bits, rel=1e-12)


def test_invalid_accounting_arguments():
    with pytest.raises(ValueError):
        storage_bits(2, 48, 1, 256, 100)
    with pytest.raises(ValueError):
        storage_bits(2, 16, 1, 256, 0)
