"""GPU parity of the 16-bit centroid storage formats (binary16, bfloat16) against the oracle.

With a 16-bit format every stored centroid is the format's round to nearest even of the
cluster's exact mean (or of the cold-start row / warm-start value it was started from), and
the residuals, codes and reconstruction are taken against those rounded values.  The checks:
  * forced: given the GPU's assignments, each stored centroid is the rounding of the exact
    mean of its stage input (computed in fp64 from X and the stored centroids), and the codes
    and scales are the oracle's encoding of the final residual;
  * the fused dequant reconstructs from the rounded tables;
  * end to end, stage by stage, against the oracle run in the same format: assignments
    agree on 99.9 % of tokens, every mismatch is a near tie (1e-3 relative distance gap),
    and the Lloyd objective is within 1e-3 relative;
  * a warm-start table is rounded once into the format (clusters left empty keep it);
  * format 0 gives the same bits as a call that never names a format.
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

FORMATS = [qvg.QVG_CENTROIDS_F16, qvg.QVG_CENTROIDS_BF16]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qbuild.build()
    qvg.load()
    torch.cuda.set_device(0)


def _run(X, C, T, bits, group, iters, seed, fmt, warm=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ckv = api.quantize(X.cuda(), C, T, bits, group, iters, seed, status=status,
                       warm=None if warm is None else torch.as_tensor(warm).cuda(),
                       centroid_format=fmt)
    x32 = api.dequantize(ckv, X.shape[1], torch.float32, status=status).cpu().numpy()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = {k: getattr(ckv, k).cpu().numpy() for k in ("codes", "scales", "pi", "centroids")}
    return ckv, g, x32


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("H,fr,gh,gw,C,T,bits,group,iters,dtype", [
    (2, 3, 20, 50, 64, 2, 2, 32, 5, torch.bfloat16),   # N = 3000
    (1, 2, 23, 29, 37, 3, 4, 16, 3, torch.float16),    # N = 1334, ragged tail
])
def test_stored_centroids_match_oracle(fmt, H, fr, gh, gw, C, T, bits, group, iters, dtype):
    X = synth.kv_tensor(200 + C, list(range(H)), 0, fr, gh, gw, dtype, "cpu")
    Xd = oracle.decode_input(X)
    ckv, g, x32 = _run(X, C, T, bits, group, iters, 9, fmt)
    assert ckv.centroid_format == fmt
    ref = oracle.quantize(Xd, C, T, bits, group, iters, 9, centroid_format=fmt)
    for h in range(H):
        cent = g["centroids"][h, 0]
        R = np.array(Xd[h], dtype=np.float64)
        for t in range(T):
            qc.check_centroids_stored(R, g["pi"][h][t], cent[t], t + 1, fmt)
            R = oracle.subtract(R, g["pi"][h][t].astype(np.int32), cent[t])
        qc.compare_codes(R, g["codes"][h], g["scales"][h], bits, group)
        qc.check_reconstruction(x32[h], g["codes"][h], g["scales"][h], g["pi"][h], cent, bits,
                                group)
        qc.check_oracle_run(Xd[h], g["pi"][h], cent, ref["pi"][h], ref["centroids"][h],
                            ref["J"][h])


@pytest.mark.parametrize("fmt", FORMATS)
def test_warm_table_is_rounded_once(fmt):
    X = synth.kv_tensor(31, [0], 0, 1, 24, 30, torch.bfloat16, "cpu")  # N = 720
    Xd = oracle.decode_input(X)
    C, T = 16, 1
    rng = np.random.default_rng(5)
    warm = Xd[0][rng.choice(X.shape[1], C, replace=False)].astype(np.float32)
    warm += rng.standard_normal(warm.shape).astype(np.float32) * np.float32(1e-3)
    # the upper half repeats the lower half: ties go to the lower index, so these clusters
    # stay empty and keep their starting value
    warm[C // 2:] = warm[:C // 2]
    _, g, _ = _run(X, C, T, 2, 32, 1, 0, fmt, warm=warm[None, None])
    cent = g["centroids"][0, 0, 0]
    np.testing.assert_array_equal(cent[C // 2:],
                                  oracle.store_centroids(warm[C // 2:].astype(np.float64), fmt))
    assert (g["pi"][0][0] < C // 2).all()
    ref = oracle.quantize(Xd, C, T, 2, 32, 1, 0, warm=warm[None, None], centroid_format=fmt)
    qc.check_oracle_run(Xd[0], g["pi"][0], g["centroids"][0, 0], ref["pi"][0],
                        ref["centroids"][0], ref["J"][0])
    qc.check_centroids_stored(Xd[0], g["pi"][0][0], cent, 1, fmt)


def test_format_0_is_the_default_path():
    X = synth.kv_tensor(7, [0, 1], 0, 2, 17, 30, torch.bfloat16, "cpu")
    a = api.quantize(X.cuda(), 16, 2, 2, 32, 3, 4)
    b = api.quantize(X.cuda(), 16, 2, 2, 32, 3, 4, centroid_format=qvg.QVG_CENTROIDS_F32)
    torch.cuda.synchronize()
    for k in ("codes", "scales", "pi", "centroids"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
