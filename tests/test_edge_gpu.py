"""GPU parity on the degenerate and extreme inputs of the method, against the oracle.

  * more stages than the unrolled kernels cover (T = 6): the generic-T paths of the
    residual, encode and dequant kernels;
  * values too large for the fp16 GEMM operands (|r| >= 60000): every cluster of such a row
    is re-scored exactly;
  * every token identical: all distances tie, so every assignment must go to the lowest
    index, and every stage after the first sees a zero residual;
  * the largest cluster count with C = N = 256: each token is its own cluster, so the
    residual and every scale are zero and the reconstruction is exact;
  * a stored cluster index >= C (a corrupted cache): flagged and clamped to C - 1.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import qvg_checks as qc
from video_kv_cache_gb300 import api
from video_kv_cache_gb300 import build as qbuild
from video_kv_cache_gb300 import qvg, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qbuild.build()
    qvg.load()
    torch.cuda.set_device(0)


def _np(ckv):
    return {k: getattr(ckv, k).cpu().numpy() for k in ("codes", "scales", "pi", "centroids")}


def _run(X, C, T, bits, group, iters, seed):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ckv = api.quantize(X.cuda(), C, T, bits, group, iters, seed, status=status)
    x32 = api.dequantize(ckv, out_dtype=torch.float32, status=status)
    torch.cuda.synchronize()
    return ckv, x32.cpu().numpy(), int(status.item())


def _check_all(X, ckv, x32, C, T, bits, group, iters, seed, min_agree=0.999):
    Xd = oracle.decode_input(X)
    g = _np(ckv)
    ref = oracle.quantize(Xd, C, T, bits, group, iters, seed)
    for h in range(X.shape[0]):
        qc.forced_check(Xd[h], g["codes"][h], g["scales"][h], g["pi"][h], g["centroids"][h, 0],
                        bits, group)
        qc.check_reconstruction(x32[h], g["codes"][h], g["scales"][h], g["pi"][h],
                                g["centroids"][h, 0], bits, group)
        qc.check_oracle_run(Xd[h], g["pi"][h], g["centroids"][h, 0], ref["pi"][h],
                            ref["centroids"][h], ref["J"][h], min_agree=min_agree)
    return g, ref


def test_six_stages_generic_paths():
    X = synth.kv_tensor(41, [0, 1], 0, 1, 20, 30, torch.bfloat16, "cpu")  # N = 600
    for bits, group in ((2, 32), (4, 16)):
        ckv, x32, st = _run(X, 8, 6, bits, group, 2, 3)
        assert st == 0
        _check_all(X, ckv, x32, 8, 6, bits, group, 2, 3)


def test_values_beyond_fp16_range_use_exact_rescoring():
    # an fp32 tensor whose channels reach +-2e5: the fp16 GEMM operands would overflow,
    # so every row must fall back to exact re-scoring of all clusters
    rng = np.random.default_rng(5)
    base = rng.standard_normal((1, 900, 128)) * 3e4
    base[0, :, 0] += rng.choice([-2e5, 2e5], size=900)
    X = torch.from_numpy(base.astype(np.float32))
    ckv, x32, st = _run(X, 16, 2, 4, 32, 3, 7)
    assert st == 0
    _check_all(X, ckv, x32, 16, 2, 4, 32, 3, 7)


def test_identical_tokens_tie_to_lowest_index():
    row = synth.kv_tensor(42, [0], 0, 1, 1, 1, torch.bfloat16, "cpu")[0, 0]
    X = row.expand(1, 513, 128).contiguous()
    ckv, x32, st = _run(X, 16, 2, 2, 32, 3, 1)
    assert st == 0
    g, ref = _check_all(X, ckv, x32, 16, 2, 2, 32, 3, 1, min_agree=1.0)
    assert (g["pi"] == 0).all()
    # stage 2 sees a zero residual, its centroids are zero, and so is every code's value
    assert (g["centroids"][0, 0, 1] == 0).all()
    assert (g["scales"] == 0).all()


def test_max_clusters_equal_tokens_is_lossless():
    X = synth.kv_tensor(43, [0, 1], 0, 1, 16, 16, torch.bfloat16, "cpu")  # N = 256
    ckv, x32, st = _run(X, 256, 1, 2, 32, 2, 9)
    assert st == 0
    g = _np(ckv)
    assert (g["scales"] == 0).all()
    np.testing.assert_array_equal(x32, oracle.decode_input(X))
    for h in range(2):
        assert sorted(g["pi"][h, 0].tolist()) == list(range(256))


def test_out_of_range_cluster_index_is_flagged_and_clamped():
    X = synth.kv_tensor(44, [0], 0, 1, 10, 30, torch.bfloat16, "cpu")  # N = 300
    C, T, bits, group = 16, 2, 2, 32
    ckv, _, st = _run(X, C, T, bits, group, 2, 5)
    assert st == 0
    ckv.pi[0, 1, 7] = 200  # a stored index >= C, as a corrupted cache could hold
    ckv.pi[0, 0, 9] = 255
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x32 = api.dequantize(ckv, out_dtype=torch.float32, status=status).cpu().numpy()
    torch.cuda.synchronize()
    assert int(status.item()) & qvg.QVG_DEV_BAD_INDEX
    g = _np(ckv)
    pi = np.minimum(g["pi"][0], C - 1)  # the documented clamp
    want = oracle.dequantize(g["codes"][0], g["scales"][0], pi, g["centroids"][0, 0], bits, group)
    S = np.abs(want) + np.abs(g["centroids"][0, 0]).max()
    assert np.all(np.abs(x32[0] - want) <= (T + 1) * np.spacing(S.astype(np.float32)))
