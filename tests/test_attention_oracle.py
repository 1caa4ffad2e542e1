"""Pins of the attention oracle (oracle/attention.py), on the CPU.

Each pin ties it to something other than its own formula:
  * torch's scaled_dot_product_attention in fp64 (a library routine);
  * closed forms: one key gives its value; all-equal scores give the mean of the values;
    a key whose score leads by hundreds gives its value exactly (the other weights
    underflow), which also fails if the scores are not shifted before the exponential;
  * invariances: permuting the keys together with their values, adding one vector to
    every key (every score of a query moves by the same amount), linearity in the values;
  * composition with the compressed cache: a cache that reconstructs X exactly
    (C = N, one cluster per token) gives the attention over X itself.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oatt


def _qkv(seed, M, N, d=128, scale_k=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((M, d)), rng.standard_normal((N, d)) * scale_k,
            rng.standard_normal((N, d)))


@pytest.mark.parametrize("M,N", [(1, 1), (3, 50), (16, 700)])
def test_matches_torch_sdpa_in_fp64(M, N):
    Q, K, V = _qkv(M + N, M, N, scale_k=2.0)
    scale = 1.0 / np.sqrt(128)
    got = oatt.attention(Q, K, V, scale)
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        scale=scale)[0].numpy()
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_one_key_gives_its_value():
    Q, K, V = _qkv(1, 4, 1)
    np.testing.assert_array_equal(oatt.attention(Q, K, V, 0.3), np.repeat(V, 4, axis=0))


def test_equal_scores_give_the_mean_value():
    _, K, V = _qkv(2, 1, 300)
    Q = np.zeros((2, 128))
    np.testing.assert_allclose(oatt.attention(Q, K, V, 1.0), np.repeat(V.mean(0, keepdims=True), 2, 0),
                               rtol=0, atol=1e-14)


def test_a_leading_key_takes_all_the_weight():
    Q, K, V = _qkv(3, 1, 40)
    K[17] = Q[0] * 10.0  # its score is about 10 |q|^2 = 1280, far above the others
    S = Q @ K.T
    assert S[0, 17] - np.delete(S[0], 17).max() > 800
    np.testing.assert_array_equal(oatt.attention(Q, K, V, 1.0)[0], V[17])


def test_invariances():
    Q, K, V = _qkv(4, 5, 200)
    s = 0.125
    O = oatt.attention(Q, K, V, s)
    perm = np.random.default_rng(0).permutation(200)
    np.testing.assert_allclose(oatt.attention(Q, K[perm], V[perm], s), O, rtol=0, atol=1e-13)
    u = np.random.default_rng(1).standard_normal(128) * 3.0
    np.testing.assert_allclose(oatt.attention(Q, K + u, V, s), O, rtol=0, atol=1e-12)
    V2 = np.random.default_rng(2).standard_normal(V.shape)
    np.testing.assert_allclose(oatt.attention(Q, K, 2.0 * V - 3.0 * V2, s),
                               2.0 * O - 3.0 * oatt.attention(Q, K, V2, s), rtol=0, atol=1e-12)


def test_exact_cache_gives_attention_over_x():
    rng = np.random.default_rng(5)
    N = 48
    X = rng.standard_normal((2, N, 128)).astype(np.float32).astype(np.float64)
    # one cluster per token: every residual is zero and the reconstruction is X itself
    ref = oracle.quantize(X, N, 1, 2, 32, 2, 11)
    caches = [{k: ref[k][h] for k in ("codes", "scales", "pi", "centroids")} for h in range(2)]
    np.testing.assert_array_equal(oatt.decode_tensor(caches[0], 2, 32), X[0])
    Q = rng.standard_normal((3, 128))
    got = oatt.attention_compressed(Q, caches[0], caches[1], 2, 32, 0.1)
    np.testing.assert_array_equal(got, oatt.attention(Q, X[0], X[1], 0.1))


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oatt.attention(np.zeros((1, 128)), np.zeros((0, 128)), np.zeros((0, 128)), 1.0)
    with pytest.raises(ValueError):
        oatt.attention(np.zeros((1, 64)), np.zeros((3, 128)), np.zeros((3, 128)), 1.0)
