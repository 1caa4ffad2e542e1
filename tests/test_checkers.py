"""The GPU parity checkers (tests/qvg_checks.py), tested on the CPU: each accepts a correct
result and rejects one with a planted error.  The correct results come from the oracle (or,
for attention, from a numpy model of the kernels' fp32 arithmetic); the errors are planted
in copies of them."""
import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oatt
from tests import attention_model
from tests import qvg_checks as qc


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


@pytest.fixture(scope="module")
def case():
    rng = np.random.default_rng(21)
    X = _bf16(rng.standard_normal((2, 700, 128)) * 2 + rng.standard_normal((2, 1, 128)) * 6)
    ref = oracle.quantize(X, 24, 2, 2, 32, 3, 4)
    return X, ref


def test_compare_codes(case):
    X, ref = case
    R = oracle.residual(X[0], ref["pi"][0], ref["centroids"][0], 2)
    codes, scales = ref["codes"][0].copy(), ref["scales"][0].copy()
    res = qc.compare_codes(R, codes, scales, 2, 32)
    assert res["code_mismatch"] == 0 and res["scale_mismatch"] == 0
    bad = codes.copy()
    bad[5, 1] ^= 0x0C  # channel 5's code (bits 2-3 of byte 1)
    with pytest.raises(AssertionError):
        qc.compare_codes(R, bad, scales, 2, 32)
    bads = scales.copy()
    bads[9, 2] ^= 0x01
    with pytest.raises(AssertionError):
        qc.compare_codes(R, codes, bads, 2, 32)


def test_check_centroids(case):
    X, ref = case
    R = X[0]
    pi = ref["pi"][0][0]
    # the fp32 rounding of the exact means passes
    C = 24
    sums = np.zeros((C, 128))
    np.add.at(sums, pi.astype(np.int64), R)
    n = np.bincount(pi, minlength=C)
    exact = np.where(n[:, None] > 0, sums / np.maximum(n, 1)[:, None], 0.0).astype(np.float32)
    qc.check_centroids(R, pi, exact, 1)
    bad = exact.copy()
    bad[3, 4] = np.nextafter(np.nextafter(bad[3, 4], np.float32(np.inf)), np.float32(np.inf))
    with pytest.raises(AssertionError):
        qc.check_centroids(R, pi, bad, 1)
    # one ulp off (the fp32 neighbour, not the rounding of the exact mean) fails too, at the
    # first stage and on a later stage's residuals
    R2 = oracle.residual(R, ref["pi"][0], ref["centroids"][0], 1)
    for stage, Rs, pis in ((1, R, pi), (2, R2, ref["pi"][0][1])):
        ns = np.bincount(pis, minlength=C)
        sums = np.zeros((C, 128))
        np.add.at(sums, pis.astype(np.int64), Rs)
        want = np.where(ns[:, None] > 0, sums / np.maximum(ns, 1)[:, None], 0.0).astype(np.float32)
        res = qc.check_centroids(Rs, pis, want, stage)
        # only means far smaller than their members fall in the band
        assert res["band"] <= 0.05 * res["entries"], res
        bad = want.copy()
        j = int(np.argmax(ns))
        k = int(np.argmax(np.abs(want[j])))
        bad[j, k] = np.nextafter(bad[j, k], np.float32(-np.inf))
        with pytest.raises(AssertionError):
            qc.check_centroids(Rs, pis, bad, stage)


def test_check_centroids_stored():
    rng = np.random.default_rng(22)
    X = _bf16(rng.standard_normal((1, 500, 128)) * 3)
    ref = oracle.quantize(X, 16, 1, 2, 32, 3, 2, centroid_format=1)
    cent = ref["centroids"][0][0]
    qc.check_centroids_stored(X[0], ref["pi"][0][0], cent, 1, 1)
    bad = cent.copy()
    bad[2, 9] = np.float32(np.nextafter(np.float16(bad[2, 9]), np.float16(np.inf)))
    with pytest.raises(AssertionError):
        qc.check_centroids_stored(X[0], ref["pi"][0][0], bad, 1, 1)


def test_check_reconstruction(case):
    X, ref = case
    args = (ref["codes"][0], ref["scales"][0], ref["pi"][0], ref["centroids"][0], 2, 32)
    x32 = oracle.dequantize(*args).astype(np.float32)
    qc.check_reconstruction(x32, *args)
    sq = oracle.e4m3_decode(ref["scales"][0])
    bad = x32.copy()
    bad[11, 40] += np.float32(0.01 * sq[11, 1] + 1e-3)
    with pytest.raises(AssertionError):
        qc.check_reconstruction(bad, *args)


def test_attention_tolerance(case):
    _, ref = case
    kc = {k: ref[k][0] for k in ("codes", "scales", "pi", "centroids")}
    vc = {k: ref[k][1] for k in ("codes", "scales", "pi", "centroids")}
    K, ek = qc.decode_with_slack(kc["codes"], kc["scales"], kc["pi"], kc["centroids"], 2, 32)
    V, ev = qc.decode_with_slack(vc["codes"], vc["scales"], vc["pi"], vc["centroids"], 2, 32)
    Q = _bf16(np.random.default_rng(3).standard_normal((6, 128)) * 2)
    scale = 128 ** -0.5
    want = oatt.attention(Q, K, V, scale)
    tol = qc.attention_tolerance(Q, K, V, ek, ev, scale)
    got = attention_model.attention_fp32(Q, K, V, scale)
    assert np.all(np.abs(got - want) <= tol)
    # a key read one row off, or one output off by a hundredth of the largest value, fails
    shifted = attention_model.attention_fp32(Q, np.roll(K, 1, axis=0), V, scale)
    assert not np.all(np.abs(shifted - want) <= tol)
    bad = got.copy()
    bad[2, 17] += 0.01 * np.abs(V).max()
    assert not np.all(np.abs(bad - want) <= tol)


def test_model_splits_match_the_library_rule():
    # the model cuts keys like the library: a multiple of 32 keys per split, at least 64,
    # about 2048 splits over all heads, every split non-empty
    for heads in (1, 3, 12, 360):
        for N in (1, 31, 32, 255, 256, 257, 1000, 32760, 32768, 280800):
            L = attention_model.split_len(N, heads)
            S = (N + L - 1) // L
            assert L % 32 == 0 and L >= 64 and (S - 1) * L < N
            assert S * heads <= max(2048, heads)
    assert attention_model.split_len(32760, 12) == 224 and attention_model.split_len(32760, 1) == 64
    assert attention_model.split_len(280800, 12) == 1664


def test_assignment_agreement(case):
    X, ref = case
    Rin = [oracle.residual(X[0], ref["pi"][0], ref["centroids"][0], t) for t in range(2)]
    same = qc.assignment_agreement(ref["pi"][0], ref["pi"][0], Rin, ref["centroids"][0])
    assert all(a["agree"] == 1.0 and a["mismatches"] == 0 for a in same)
    moved = ref["pi"][0].copy()
    moved[1, :7] = (moved[1, :7] + 1) % 24
    res = qc.assignment_agreement(moved, ref["pi"][0], Rin, ref["centroids"][0])
    assert res[0]["mismatches"] == 0 and res[1]["mismatches"] == 7 and res[1]["max_gap"] > 0
