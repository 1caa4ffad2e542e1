"""Oracle of attention read straight from a compressed cache.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``, the package smoke
check and the benchmark's CPU-baseline leg may use it.

What it computes.  The fused reconstruction exists to feed attention without writing the
rebuilt cache back to memory ("Quant VideoGen" notes page, Algorithm-System Co-design: the
cache is reconstructed on the fly for attention).  The pages do not restate attention; this
is the standard scaled dot-product form.  A query q against keys k_j and values v_j
(j < N) gives o = sum_j p_j v_j, where p = softmax(scale * q.k_j) over j.  The keys and
values are the oracle's own fp64 decode of the compressed tensors: the final residual's
codes plus every stage's assigned centroid.

Plain numpy in fp64.  The scores are shifted by their maximum before the exponential.  That
leaves the softmax unchanged and keeps exp from overflowing.
"""
from __future__ import annotations

import numpy as np

from . import dequantize


def attention(Q, K, V, scale: float) -> np.ndarray:
    """Softmax attention of queries Q [M][d] over keys K [N][d] and values V [N][d], fp64."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if Q.ndim != 2 or K.ndim != 2 or V.shape != K.shape or Q.shape[1] != K.shape[1]:
        raise ValueError("need Q [M][d], K [N][d], V [N][d]")
    if K.shape[0] == 0:
        raise ValueError("attention over no keys is undefined")
    S = float(scale) * (Q @ K.T)
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    return (P @ V) / P.sum(axis=1, keepdims=True)


def decode_tensor(cache: dict, bits: int, group: int, scheme: int = 0) -> np.ndarray:
    """fp64 reconstruction of one compressed tensor given as a dict of its codes [N][..],
    scales [N][..], pi [T][N] and centroids [T][C][d] (one table)."""
    return dequantize(cache["codes"], cache["scales"], cache["pi"], cache["centroids"], bits,
                      group, scheme)


def attention_compressed(Q, k_cache: dict, v_cache: dict, bits: int, group: int, scale: float,
                         scheme: int = 0) -> np.ndarray:
    """Attention of Q [M][d] over the keys and values rebuilt from two compressed tensors."""
    K = decode_tensor(k_cache, bits, group, scheme)
    V = decode_tensor(v_cache, bits, group, scheme)
    return attention(Q, K, V, scale)
