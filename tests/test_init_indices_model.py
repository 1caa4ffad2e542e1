"""The cold start's sparse shuffle, modelled on the CPU.

The oracle draws the seeded start rows with a partial Fisher-Yates shuffle over a full
permutation array of 0..N-1.  The GPU kernel (k_init_indices) keeps only the touched
positions: positions below C in an array, the others in a 1024-slot open-addressing table
(multiplicative hash, linear probing), and draws all C SplitMix64 outputs up front from the
generator's state + k * gamma.  This test restates that algorithm in Python integers and
checks that it returns the oracle's indices for random and edge-case (N, C): C = N,
C = N - 1, C = 1, N up to 2^22 (and distinct, in-range indices up to N = 2^31 - 1), and
a 16-slot table that forces long probe chains."""
import numpy as np
import pytest

import oracle

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def _splitmix_output(state):
    z = (state + GAMMA) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def sparse_init_indices(seed, tensor_id, stage, N, C, slots=1024):
    state0 = (seed ^ ((tensor_id * GAMMA) & M64) ^ stage) & M64
    pick = [x + _splitmix_output((state0 + x * GAMMA) & M64) % (N - x) for x in range(C)]
    lo = list(range(C))
    keys, vals = [-1] * slots, [0] * slots
    out = []
    for j in range(C):
        k = pick[j]
        if k < C:
            vk = lo[k]
        else:
            slot = (((k * 2654435761) & 0xFFFFFFFF) >> 22) & (slots - 1)
            while keys[slot] != -1 and keys[slot] != k:
                slot = (slot + 1) & (slots - 1)
            vk = vals[slot] if keys[slot] == k else k
        vj = lo[j]
        out.append(vk)
        if k < C:
            lo[k] = vj
        else:
            keys[slot], vals[slot] = k, vj
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("N,C", [(1, 1), (2, 2), (256, 256), (257, 256), (300, 1),
                                  (4096, 64), (32760, 256), (4680, 256), (1 << 22, 256),
                                  ((1 << 31) - 1, 256)])
def test_matches_the_oracle(N, C):
    for seed, tid, stage in ((0, 0, 1), (12345, 7, 2), (2 ** 63 + 5, 719, 4)):
        got = sparse_init_indices(seed, tid, stage, N, C)
        assert len(set(got.tolist())) == C and got.min() >= 0 and got.max() < N
        if N <= (1 << 22):  # the oracle holds the whole permutation (8 N bytes)
            assert np.array_equal(got, oracle.init_indices(seed, tid, stage, N, C))


def test_random_sizes():
    rng = np.random.default_rng(0)
    for _ in range(300):
        C = int(rng.integers(1, 257))
        N = int(C + rng.integers(0, 5000))
        seed, tid, stage = int(rng.integers(0, 2 ** 63)), int(rng.integers(0, 1000)), int(rng.integers(1, 9))
        assert np.array_equal(sparse_init_indices(seed, tid, stage, N, C),
                              oracle.init_indices(seed, tid, stage, N, C))


def test_colliding_hash_keys():
    # a table of 16 slots forces long probe chains; the result must not change
    rng = np.random.default_rng(1)
    for _ in range(50):
        C = int(rng.integers(1, 9))
        N = int(C + rng.integers(1, 100000))
        args = (int(rng.integers(0, 2 ** 63)), 3, 1, N, C)
        assert np.array_equal(sparse_init_indices(*args, slots=16), oracle.init_indices(*args))
