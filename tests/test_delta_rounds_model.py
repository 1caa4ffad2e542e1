"""The bookkeeping of the Lloyd rounds that fold in only the tokens that changed cluster,
modelled on the CPU with integer values (so every sum is exact).

A stage's first round sorts every token by its cluster.  A later round sorts, for every
token whose cluster changed since the previous round, a leave item keyed by its old
cluster (its row negated) and an enter item keyed by its new one.  The counting sort works
on blocks of 256 tokens: the block histogram counts both kinds; the scatter places a
block's items of one cluster leave items first, then enter items, each kind in token order,
with a position

    leave: blockoff[b][j] + (leave items of j in the block's earlier warps) + (rank in warp)
    enter: blockoff[b][j] + (all leave items of j in the block)
                          + (enter items of j in the block's earlier warps) + (rank in warp)

where blockoff[b][j] is the offset of cluster j plus its items in the blocks before b.
The chunk sums and the finalize's choice of pieces are the full round's (see
test_cluster_sum_slots_model.py); the finalize then adds the pieces to the total the
previous round kept and sets the member count to kept + items - 2 * leaves.

The test replays several rounds with random reassignments (few tokens moving, most, none,
a cluster emptied and refilled, ragged token counts) and checks after every round that
  * the scatter's positions are a bijection onto the round's items, in the sort's order;
  * every cluster's kept total is the exact sum of its members' values, and its count the
    number of its members."""
import numpy as np
import pytest

from tests.test_cluster_sum_slots_model import _chunk_sums, _finalize

BLOCK, WARP = 256, 32


def _items(pi, pi_prev, delta):
    """(token, key, is_leave) of the round's items, and the per-key leave counts."""
    out = []
    for i, j in enumerate(pi):
        if not delta:
            out.append((i, int(j), False))
        elif pi_prev[i] != j:
            out.append((i, int(pi_prev[i]), True))
            out.append((i, int(j), False))
    return out


def _positions(items, N, C):
    """The scatter's positions, computed by the kernel's formula."""
    nsb = (N + BLOCK - 1) // BLOCK
    hist = np.zeros((nsb, C), np.int64)
    for i, j, _ in items:
        hist[i // BLOCK, j] += 1
    counts = hist.sum(0)
    offs = np.concatenate([[0], np.cumsum(counts)[:-1]])
    blockoff = offs[None, :] + np.cumsum(hist, 0) - hist          # exclusive over blocks
    nw = BLOCK // WARP
    wl = np.zeros((nsb, nw, C), np.int64)
    we = np.zeros((nsb, nw, C), np.int64)
    for i, j, leave in items:
        (wl if leave else we)[i // BLOCK, (i % BLOCK) // WARP, j] += 1
    pos = []
    for i, j, leave in items:
        b, w, lane = i // BLOCK, (i % BLOCK) // WARP, i % WARP
        w0 = b * BLOCK + w * WARP  # first token of the warp
        same = [t for (t, jj, lv) in items if jj == j and lv == leave and w0 <= t < i]
        rank = len(same)           # earlier lanes of the warp with the same key and kind
        if leave:
            p = blockoff[b, j] + wl[b, :w, j].sum() + rank
        else:
            p = blockoff[b, j] + wl[b, :, j].sum() + we[b, :w, j].sum() + rank
        pos.append(int(p))
    return pos, counts, offs


def _round(pi, pi_prev, delta, vals, kept_tot, kept_n, C):
    N = len(pi)
    items = _items(pi, pi_prev, delta)
    pos, counts, offs = _positions(items, N, C)
    n_items = len(items)
    assert sorted(pos) == list(range(n_items)), "positions are not a bijection"
    # the sort's order: by key, then block, leave items before enter items, then token
    want_order = sorted(range(n_items), key=lambda q: (items[q][1], items[q][0] // BLOCK,
                                                       0 if items[q][2] else 1, items[q][0]))
    assert [pos[q] for q in want_order] == list(range(n_items))
    keys = np.zeros(n_items, np.int64)
    signed = np.zeros(n_items, np.int64)
    for q, (i, j, leave) in enumerate(items):
        keys[pos[q]] = j
        signed[pos[q]] = -vals[i] if leave else vals[i]
    leaves = np.zeros(C, np.int64)
    for i, j, leave in items:
        if leave:
            leaves[j] += 1
    if n_items:
        own, piece = _chunk_sums(keys, signed, C)
        got = _finalize(counts, offs, own, piece)
    else:
        got = {}
    tot = kept_tot.copy() if delta else np.zeros(C, np.int64)
    n = kept_n + counts - 2 * leaves if delta else counts.copy()
    for j, s in got.items():
        tot[j] += s
    tot[n == 0] = 0  # an emptied cluster's total restarts at zero
    return tot, n


def _run(N, C, moves, seed):
    rng = np.random.default_rng(seed)
    vals = rng.integers(-10**6, 10**6, N)
    pi = rng.integers(0, C, N)
    pi_prev = np.zeros(N, np.int64)
    tot, n = np.zeros(C, np.int64), np.zeros(C, np.int64)
    for r, frac in enumerate(moves):
        if r > 0:
            pi = pi.copy()
            sel = rng.random(N) < frac
            pi[sel] = rng.integers(0, C, int(sel.sum()))
        tot, n = _round(pi, pi_prev, r > 0, vals, tot, n, C)
        want_tot = np.bincount(pi, weights=vals, minlength=C).astype(np.int64)
        want_n = np.bincount(pi, minlength=C)
        assert np.array_equal(n, want_n), ("counts", r)
        assert np.array_equal(tot, want_tot), ("totals", r)
        pi_prev = pi


@pytest.mark.parametrize("N,C,moves", [
    (300, 7, [1.0, 0.5, 0.1, 0.02, 0.0, 0.3]),     # ragged last block, few clusters
    (600, 40, [1.0, 0.9, 0.05, 0.05, 0.01]),       # most tokens move once, then few
    (257, 3, [1.0, 0.0, 1.0, 0.0]),                # rounds with nothing moving
    (520, 64, [1.0, 0.2, 0.2, 0.2]),               # many clusters with few members
])
def test_rounds_keep_exact_totals(N, C, moves):
    _run(N, C, moves, seed=N + C)


def test_cluster_emptied_and_refilled():
    N, C = 300, 5
    rng = np.random.default_rng(1)
    vals = rng.integers(-1000, 1000, N)
    pi0 = rng.integers(0, C, N)
    pi1 = np.where(pi0 == 2, 3, pi0)          # cluster 2 empties
    pi2 = pi1.copy()
    pi2[::7] = 2                              # and fills again
    tot, n = _round(pi0, np.zeros(N, np.int64), False, vals, np.zeros(C, np.int64),
                    np.zeros(C, np.int64), C)
    tot, n = _round(pi1, pi0, True, vals, tot, n, C)
    assert n[2] == 0 and tot[2] == 0
    tot, n = _round(pi2, pi1, True, vals, tot, n, C)
    assert np.array_equal(tot, np.bincount(pi2, weights=vals, minlength=C).astype(np.int64))
    assert np.array_equal(n, np.bincount(pi2, minlength=C))
