"""Named settings of the method and the storage accounting of a compressed cache.

Presets ("Quant VideoGen" explainer page, results: the block-size trade-off):
  * ``qvg``     -- one smoothing stage and 64-channel scale groups, the setting that
    maximises compression;
  * ``qvg_pro`` -- four stages and 16-channel groups, the setting that maximises fidelity.
Both use INT2 codes with FP8 E4M3 group scales, the pages' headline precision, and C = 256
centroids per stage.  They are parameter choices: the library takes any (C, T, bits,
group) in its supported ranges.

Storage accounting (same page, compression and metadata overhead).  A token of d channels
costs, in bits:
  * codes:     d * bits
  * scales:    8 * d / group (one E4M3 byte per group)
  * pi:        8 * T (one cluster byte per stage)
  * centroids: T * C * d * centroid_bits, once per tensor, so N tokens share it
The compression ratio is the 16-bit input over that total.  The library keeps its centroid
tables as fp32 arrays (centroid_bits = 32, what ``cache_bytes`` counts).  The pages' ratios
count 16-bit centroids: with a 16-bit centroid format (qvg.QVG_CENTROIDS_F16 / _BF16) every
stored value is representable in 16 bits, so a consumer that narrows the tables stores what
``storage_bits(..., centroid_bits=16)`` counts.
"""
from __future__ import annotations

from dataclasses import dataclass

D = 128


@dataclass(frozen=True)
class Preset:
    name: str
    C: int
    T: int
    bits: int
    group: int


PRESETS = {
    "qvg": Preset("qvg", C=256, T=1, bits=2, group=64),
    "qvg_pro": Preset("qvg_pro", C=256, T=4, bits=2, group=16),
}


def storage_bits(bits: int, group: int, T: int, C: int, N: int, centroid_bits: int = 32,
                 d: int = D) -> dict:
    """Bits per element of each part of a compressed tensor of N tokens, their total, the
    compression ratio against a 16-bit input and the codes' share of the storage."""
    if N <= 0 or d % group:
        raise ValueError("need N > 0 and d a multiple of group")
    parts = {
        "codes": float(bits),
        "scales": 8.0 / group,
        "pi": 8.0 * T / d,
        "centroids": float(T * C * centroid_bits) / N,
    }
    total = sum(parts.values())
    return {"bits_per_element": parts, "total_bits_per_element": total,
            "compression_ratio": 16.0 / total, "codes_share": parts["codes"] / total}


def cache_bytes(ckv, N: int) -> int:
    """Bytes that a CompressedKV holding N tokens per tensor (one table slot) occupies:
    the codes, scales and pi of N tokens and every tensor's centroid tables."""
    H = ckv.codes.shape[0]
    per_token = (ckv.codes.shape[2] * ckv.codes.element_size() +
                 ckv.scales.shape[2] * ckv.scales.element_size() +
                 ckv.pi.shape[1] * ckv.pi.element_size())
    tables = ckv.centroids[:, :1].numel() * ckv.centroids.element_size()
    return H * N * per_token + tables
