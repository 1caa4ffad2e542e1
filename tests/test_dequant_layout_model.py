"""The fused dequant's staged-table layout, modelled on the CPU.

A staged table row holds W / 4 chunks of 16 bytes; logical chunk c of row r is stored at
chunk swz(r, c) = c ^ ((c >> 3) & 3) ^ ((r & 1) << 1).  Checked here:
  * correctness: for every row, swz is a permutation of the row's chunks (no two logical
    chunks share a slot), for W = 32, 64 and 128;
  * the bank claims: the lanes of one token read chunks 4 sub + k (sub = 0 .. W/16 - 1) of
    their row for k = 0..3.  At W = 128 a quarter-warp is one token and its eight reads
    fall in eight distinct 16-byte bank groups; at W = 64 it is two tokens, disjoint when
    their rows differ in parity; at W = 32 (four tokens) rows of different parity are
    still disjoint."""
import pytest


def swz(r, c):
    return c ^ ((c >> 3) & 3) ^ ((r & 1) << 1)


@pytest.mark.parametrize("W", [32, 64, 128])
def test_swizzle_is_a_permutation_of_each_row(W):
    wq = W // 4
    for r in range(8):
        slots = [swz(r, c) for c in range(wq)]
        assert sorted(slots) == list(range(wq))


def _groups(r, W, subs, k):
    """16-byte bank groups (address mod 8 chunks) read by the lanes sub of a token on row r."""
    wq = W // 4
    return [(r * wq + swz(r, 4 * sub + k)) % 8 for sub in subs]


def test_one_token_per_quarter_warp_at_w128():
    # 8 lanes of one token read chunks 4 l + k, l = 0..7: eight distinct groups on any row
    for r in range(64):
        for k in range(4):
            assert len(set(_groups(r, 128, range(8), k))) == 8


def test_two_tokens_per_quarter_warp_at_w64():
    # 4 lanes per token: rows of different parity read disjoint groups (8 in all); the
    # same row is one address per lane pair (a broadcast)
    for ra in range(32):
        for rb in range(32):
            for k in range(4):
                ga, gb = _groups(ra, 64, range(4), k), _groups(rb, 64, range(4), k)
                assert len(set(ga)) == 4 and len(set(gb)) == 4
                if (ra ^ rb) & 1:
                    assert not set(ga) & set(gb)


def test_tokens_of_different_parity_are_disjoint_at_w32():
    # 2 lanes per token, 4 tokens per quarter-warp: a token's two reads are distinct and
    # tokens on rows of different parity never share a group (same-parity rows may)
    for ra in range(32):
        for rb in range(32):
            for k in range(4):
                ga, gb = _groups(ra, 32, range(2), k), _groups(rb, 32, range(2), k)
                assert len(set(ga)) == 2
                if (ra ^ rb) & 1:
                    assert not set(ga) & set(gb)
