"""GPU parity of qvg_attention (attention read straight from the compressed cache) against
the oracle.

The oracle side is oracle/attention.py over the oracle's fp64 decode of the very cache the
GPU wrote (the compression itself is checked elsewhere).  The bound is
qvg_checks.attention_tolerance, derived from the fp32 arithmetic of the scores, the softmax
and the sums.  Cases span several 32-key tiles and several splits, with ragged ends:
  * keys and values interleaved in one cache (tensor 2h and 2h + 1) and in two caches;
  * INT2 and INT4, both integer grids, T = 0 .. 3, bf16 / fp16 / fp32 queries, M = 1 .. 16;
  * one key: the output is the fp32 reconstruction of its value, bit for bit;
  * chunked caches with one centroid table per chunk;
  * 16-bit outputs are the round to nearest even of the fp32 output;
  * a full 32760-token head pair, on sampled channels of every query.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oatt
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


def _np(ckv, h):
    return {k: getattr(ckv, k)[h].cpu().numpy() for k in ("codes", "scales", "pi")} | \
        {"centroids": ckv.centroids[h, 0].cpu().numpy()}


def _queries(seed, H, M, dtype):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((H, M, 128), generator=g) * 2.0).to(dtype)


def _check_head(O, Qh, kc, vc, bits, group, scheme, scale):
    K, ek = qc.decode_with_slack(kc["codes"], kc["scales"], kc["pi"], kc["centroids"], bits,
                                 group, scheme)
    V, ev = qc.decode_with_slack(vc["codes"], vc["scales"], vc["pi"], vc["centroids"], bits,
                                 group, scheme)
    want = oatt.attention(Qh, K, V, scale)
    tol = qc.attention_tolerance(Qh, K, V, ek, ev, scale)
    err = np.abs(np.asarray(O, dtype=np.float64) - want)
    if not np.all(err <= tol):
        m, c = np.argwhere(err > tol)[0]
        raise AssertionError("query %d channel %d: got %r want %r tol %r" %
                             (m, c, O[m, c], want[m, c], tol[m, c]))
    return float((err / tol).max())


CASES = [
    # heads, frames, gh, gw, C, T, bits, group, scheme, M, q dtype
    (2, 2, 20, 25, 32, 2, 2, 32, 0, 5, torch.bfloat16),    # N = 1000: 4 splits, ragged tile
    (1, 3, 17, 23, 16, 1, 4, 16, 0, 16, torch.float16),    # N = 1173
    (2, 1, 9, 13, 5, 3, 2, 64, 1, 1, torch.float32),       # N = 117 < one split
    (1, 2, 16, 40, 64, 0, 4, 64, 1, 3, torch.bfloat16),    # T = 0, N = 1280
]


@pytest.mark.parametrize("case", CASES)
def test_attention_interleaved_cache_matches_oracle(case):
    Hh, fr, gh, gw, C, T, bits, group, scheme, M, qdt = case
    X = synth.kv_tensor(40 + C, list(range(2 * Hh)), 0, fr, gh, gw, torch.bfloat16, "cuda")
    N = X.shape[1]
    ckv = api.quantize(X, C, T, bits, group, 3, 5, qscheme=scheme)
    Q = _queries(C + M, Hh, M, qdt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 128 ** -0.5
    O = api.attention(Q.cuda(), ckv, scale=scale, N=N, k_first=0, v_first=1, tensor_step=2,
                      status=status).cpu().numpy()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Qd = Q.double().numpy()
    for h in range(Hh):
        _check_head(O[h], Qd[h], _np(ckv, 2 * h), _np(ckv, 2 * h + 1), bits, group, scheme, scale)


def test_attention_separate_caches_and_fp32_reconstruction():
    X = synth.kv_tensor(77, list(range(6)), 0, 2, 30, 31, torch.bfloat16, "cuda")  # N = 1860
    N = X.shape[1]
    kcache = api.quantize(X[:3].contiguous(), 48, 2, 2, 32, 3, 1)
    vcache = api.quantize(X[3:].contiguous(), 48, 2, 2, 32, 3, 2)
    Q = _queries(3, 3, 8, torch.bfloat16)
    scale = 0.05
    O = api.attention(Q.cuda(), kcache, vcache, scale=scale, N=N).cpu().numpy()
    Qd = Q.double().numpy()
    # the same result against attention over the library's own fp32 reconstruction
    K32 = api.dequantize(kcache, N, torch.float32).cpu().numpy().astype(np.float64)
    V32 = api.dequantize(vcache, N, torch.float32).cpu().numpy().astype(np.float64)
    for h in range(3):
        _check_head(O[h], Qd[h], _np(kcache, h), _np(vcache, h), 2, 32, 0, scale)
        zero = np.zeros_like(K32[h])
        tol = qc.attention_tolerance(Qd[h], K32[h], V32[h], zero, zero, scale)
        assert np.all(np.abs(O[h] - oatt.attention(Qd[h], K32[h], V32[h], scale)) <= tol)


def test_one_key_gives_the_reconstructed_value_exactly():
    X = synth.kv_tensor(5, [0, 1], 0, 1, 12, 12, torch.bfloat16, "cuda")
    ckv = api.quantize(X, 8, 2, 2, 32, 2, 3)
    Q = _queries(1, 1, 4, torch.float32).cuda()
    O = api.attention(Q, ckv, N=1, k_first=0, v_first=1, tensor_step=2)
    v32 = api.dequantize(ckv, None, torch.float32)[1, 0]
    assert torch.equal(O[0], v32.expand(4, 128))


def test_chunked_tables():
    # two chunks of 600 tokens quantized into one cache, one centroid table each
    X = synth.kv_tensor(9, [0, 1], 0, 2, 20, 30, torch.bfloat16, "cuda")  # N = 1200
    L = 600
    out = api.allocate(2, 1200, 24, 2, 2, 32, 2, "cuda")
    for c in range(2):
        api.quantize(X[:, c * L:(c + 1) * L].contiguous(), 24, 2, 2, 32, 3, 4, out=out,
                     token_offset=c * L, table_index=c)
    Q = _queries(11, 1, 2, torch.bfloat16)
    O = api.attention(Q.cuda(), out, N=1200, chunk_len=L, k_first=0, v_first=1,
                      tensor_step=2).cpu().numpy()
    # the oracle decodes each chunk with its own table
    K, V, ek, ev = [], [], [], []
    for c in range(2):
        for h, (dst, eps) in ((0, (K, ek)), (1, (V, ev))):
            sl = slice(c * L, (c + 1) * L)
            x, e = qc.decode_with_slack(out.codes[h, sl].cpu().numpy(),
                                        out.scales[h, sl].cpu().numpy(),
                                        out.pi[h, :, sl].cpu().numpy(),
                                        out.centroids[h, c].cpu().numpy(), 2, 32)
            dst.append(x)
            eps.append(e)
    K, V, ek, ev = (np.concatenate(a) for a in (K, V, ek, ev))
    Qd = Q.double().numpy()[0]
    want = oatt.attention(Qd, K, V, 128 ** -0.5)
    tol = qc.attention_tolerance(Qd, K, V, ek, ev, 128 ** -0.5)
    assert np.all(np.abs(O[0] - want) <= tol)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_16_bit_output_is_the_rounded_fp32_output(dtype):
    X = synth.kv_tensor(13, [0, 1, 2, 3], 0, 2, 16, 20, torch.bfloat16, "cuda")
    ckv = api.quantize(X, 16, 1, 4, 32, 2, 6)
    Q = _queries(2, 2, 6, torch.bfloat16).cuda()
    o32 = api.attention(Q, ckv, k_first=0, v_first=1, tensor_step=2)
    o16 = api.attention(Q, ckv, k_first=0, v_first=1, tensor_step=2, out_dtype=dtype)
    qc.check_rounded_output(o16.cpu(), o32.cpu().numpy(), dtype)


def test_full_size_head_pair_on_sampled_channels():
    X = synth.kv_tensor(2, [0, 1], 0, 7, 90, 52, torch.bfloat16, "cuda")  # N = 32760
    N = X.shape[1]
    ckv = api.quantize(X, 256, 2, 2, 32, 4, 1)
    Q = _queries(8, 1, 16, torch.bfloat16)
    O = api.attention(Q.cuda(), ckv, N=N, k_first=0, v_first=1, tensor_step=2).cpu().numpy()
    kc, vc = _np(ckv, 0), _np(ckv, 1)
    K, ek = qc.decode_with_slack(kc["codes"], kc["scales"], kc["pi"], kc["centroids"], 2, 32)
    V, ev = qc.decode_with_slack(vc["codes"], vc["scales"], vc["pi"], vc["centroids"], 2, 32)
    check_sampled_channels(O[0], Q.double().numpy()[0], K, V, ek, ev, 128 ** -0.5)


def check_sampled_channels(O, Qd, K, V, ek, ev, scale, n_cols=24):
    # the oracle's attention over every channel; the comparison on a seeded sample of them
    cols = np.random.default_rng(0).choice(128, n_cols, replace=False)
    want = oatt.attention(Qd, K, V, scale)[:, cols]
    tol = qc.attention_tolerance(Qd, K, V, ek, ev, scale)[:, cols]
    assert np.all(np.abs(np.asarray(O, dtype=np.float64)[:, cols] - want) <= tol)
