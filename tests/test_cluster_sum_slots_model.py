"""The bookkeeping of the cluster sums, modelled on the CPU.

After the counting sort, the sorted positions are cut into chunks of 32.  Within a chunk
each run of one cluster is summed; the run's sum goes to
  * the cluster's own slot when the run is the whole cluster (it neither continues from the
    previous chunk nor into the next one),
  * else the chunk's slot 0 when the run starts the chunk, or its slot 1 otherwise.
The finalize step then takes, for cluster j with count n and first sorted position off, the
cluster's own slot if it lies in one chunk, else one piece per chunk it spans: slot 1 of
its first chunk unless it starts exactly at that chunk's start (slot 0), and slot 0 of every
later chunk.

This test replays both rules (with integer values, so the sums are exact) over random
cluster sizes and over the awkward ones -- clusters of exactly 32 or 64 starting on a chunk
boundary, single tokens at chunk edges, clusters spanning many chunks, empty clusters, a
ragged last chunk -- and checks that every cluster's total comes out right and that no slot
is written twice."""
import numpy as np
import pytest

CHUNK = 32


def _chunk_sums(cl_sorted, vals_sorted, C):
    N = len(cl_sorted)
    nchunk = (N + CHUNK - 1) // CHUNK
    own, piece = {}, {}
    for k in range(nchunk):
        lo, hi = k * CHUNK, min(N, (k + 1) * CHUNK)
        c_prev = cl_sorted[lo - 1] if lo > 0 else -1
        c_next = cl_sorted[hi] if hi < N else -1
        start = lo
        while start < hi:
            end = start
            while end < hi and cl_sorted[end] == cl_sorted[start]:
                end += 1
            c = cl_sorted[start]
            s = int(vals_sorted[start:end].sum())
            run_start, run_end, nk = start - lo, end - lo, hi - lo
            whole = (run_start > 0 or c_prev != c) and (run_end < nk or c_next != c)
            key = c if whole else (k, 0 if run_start == 0 else 1)
            target = own if whole else piece
            assert key not in target, ("slot written twice", key)
            target[key] = s
            start = end
    return own, piece


def _finalize(counts, offs, own, piece):
    out = {}
    for j, (n, off) in enumerate(zip(counts, offs)):
        if n == 0:
            continue
        a, b = off // CHUNK, (off + n - 1) // CHUNK
        if a == b:
            out[j] = own[j]
        else:
            out[j] = sum(piece[(kk, 1 if (kk == a and off != a * CHUNK) else 0)]
                         for kk in range(a, b + 1))
    return out


def _check(sizes):
    C = len(sizes)
    pi = np.repeat(np.arange(C), sizes)
    rng = np.random.default_rng(len(pi))
    pi = rng.permutation(pi)                   # tokens in any order
    vals = rng.integers(-1000, 1000, len(pi))
    order = np.argsort(pi, kind="stable")      # the stable counting sort
    counts = np.bincount(pi, minlength=C)
    offs = np.concatenate([[0], np.cumsum(counts)[:-1]])
    own, piece = _chunk_sums(pi[order], vals[order], C)
    got = _finalize(counts, offs, own, piece)
    want = np.bincount(pi, weights=vals, minlength=C).astype(np.int64)
    for j in range(C):
        if counts[j]:
            assert got[j] == want[j], (j, sizes)


@pytest.mark.parametrize("sizes", [
    [32, 32, 32],                  # clusters exactly filling chunks
    [64, 1, 31, 32],               # spans two chunks from a boundary; singles at edges
    [1, 63, 0, 0, 1, 95, 3],       # empty clusters; long spans starting mid-chunk
    [31, 2, 31, 2, 31],            # runs crossing every boundary by one
    [200],                         # one cluster, many chunks, ragged end
    [5] * 13,                      # many small runs per chunk, ragged end
    [0, 0, 40, 0],                 # empty clusters before and after
])
def test_awkward_cluster_sizes(sizes):
    _check(sizes)


def test_random_cluster_sizes():
    rng = np.random.default_rng(0)
    for _ in range(300):
        C = int(rng.integers(1, 60))
        sizes = rng.choice([0, 1, 2, 31, 32, 33, 64], size=C) * (rng.random(C) < 0.5) + \
            rng.integers(0, 70, C) * (rng.random(C) < 0.5)
        if sizes.sum() == 0:
            continue
        _check(list(sizes))
