"""GPU parity at the full workload sizes, in the launch configuration the benchmark times.

The whole workload runs on the GPU through the C ABI; the oracle then checks sampled
tensors (and, for the assignment, sampled tokens) one by one:
  * forced mode on each sampled tensor: given the GPU's assignments, every stage's
    centroids are the exact means and the codes / scales are the exact encoding of the
    final residual (bit-exact outside the rounding bands);
  * the fp32 reconstruction of each sampled tensor against the oracle's decode;
  * qvg_reassign's pi^(T) on sampled tokens against the fp64 argmin over the stored
    centroids: equal, or a tie within fp32 rounding;
  * whole tensors through the oracle's own Lloyd iterations, stage by stage: one tensor of
    the 1.3B layer, and the first head's key and value tensors of the 13B-class shape
    (65536 tokens, four stages), each to the full bar (99.9 % agreement per stage, every
    mismatch within a 1e-3 relative distance gap, objective within 1e-3).
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


def _np(t):
    return t.cpu().numpy()


def _check_reassign_sample(X, ckv, h, T, n_tokens, seed):
    """pi^(T) of tensor h (just rewritten by qvg_reassign) on sampled tokens against the
    fp64 argmin over the stored stage-T centroids."""
    rng = np.random.default_rng(seed)
    N = X.shape[1]
    rows = np.sort(rng.choice(N, size=min(n_tokens, N), replace=False))
    Xd = oracle.decode_input(X[h, torch.from_numpy(rows)].cpu().unsqueeze(0))[0]
    pi = _np(ckv.pi[h, :, torch.from_numpy(rows).cuda()])
    cent = _np(ckv.centroids[h, 0])
    R = oracle.residual(Xd, pi, cent, T - 1)
    pi_o, d_o = oracle.assign(R, cent[T - 1])
    got = pi[T - 1].astype(np.int64)
    mism = np.flatnonzero(got != pi_o)
    for i in mism:
        dg = ((R[i] - cent[T - 1][got[i]].astype(np.float64)) ** 2).sum()
        assert dg - d_o[i] <= 2.0 ** -20 * max(d_o[i], 1e-30), (h, rows[i], dg, d_o[i])
    return len(mism)


def _forced_and_reconstruction(X, ckv, xhat32, h, bits, group):
    Xd = oracle.decode_input(X[h:h + 1].cpu())[0]
    codes, scales = _np(ckv.codes[h]), _np(ckv.scales[h])
    pi, cent = _np(ckv.pi[h]), _np(ckv.centroids[h, 0])
    res = qc.forced_check(Xd, codes, scales, pi, cent, bits, group)
    qc.check_reconstruction(_np(xhat32[h]), codes, scales, pi, cent, bits, group)
    return res, Xd


def _run_full(w):
    dev = torch.device("cuda")
    X = w.make(dev)
    H, N = X.shape[:2]
    out = api.allocate(H, N, w.C, w.T, w.bits, w.group, device=dev)
    ws = api.new_workspace(H, N, w.C, w.T, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    api.quantize(X, w.C, w.T, w.bits, w.group, w.iters, w.seed, out=out, workspace=ws,
                 status=status)
    xhat32 = api.dequantize(out, N, torch.float32, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status %#x" % int(status.item())
    return X, out, ws, xhat32


def test_layer_1p3b_full_size():
    w = synth.workload("layer_1p3b_32760")
    X, ckv, ws, xhat32 = _run_full(w)
    H = X.shape[0]
    # a key and a value tensor, first and last of the batch
    for h in (0, H - 1):
        _forced_and_reconstruction(X, ckv, xhat32, h, w.bits, w.group)
    # one whole tensor through the oracle's own Lloyd iterations
    h = 0
    Xd = oracle.decode_input(X[h:h + 1].cpu())
    ref = oracle.quantize(Xd, w.C, w.T, w.bits, w.group, w.iters, w.seed, tensor_id_base=h)
    qc.check_oracle_run(Xd[0], _np(ckv.pi[h]), _np(ckv.centroids[h, 0]), ref["pi"][0],
                        ref["centroids"][0], ref["J"][0])
    # the tensor-core assignment at full size: reassign, then sampled tokens
    api.reassign(X, ckv, w.iters, ws, w.seed)
    torch.cuda.synchronize()
    for h in (0, 7, H - 1):
        _check_reassign_sample(X, ckv, h, w.T, 3000, seed=h)


def test_dit13b_full_size():
    w = synth.workload("dit13b_65536")
    X, ckv, ws, xhat32 = _run_full(w)
    H = X.shape[0]
    for h in (0, H - 1):
        res, _ = _forced_and_reconstruction(X, ckv, xhat32, h, w.bits, w.group)
        assert len(res["stages"]) == 4
    del xhat32
    # the first head's key and value tensors, whole (65536 tokens, four stages of eight
    # Lloyd rounds each), through the oracle's own independent run: every stage to the full
    # bar (99.9 % agreement, every mismatch a near tie, objective within 1e-3)
    Xd = oracle.decode_input(X[0:2].cpu())
    ref = oracle.quantize(Xd, w.C, w.T, w.bits, w.group, w.iters, w.seed, tensor_id_base=0,
                          nthreads=2)
    for h in (0, 1):
        qc.check_oracle_run(Xd[h], _np(ckv.pi[h]), _np(ckv.centroids[h, 0]), ref["pi"][h],
                            ref["centroids"][h], ref["J"][h])
    del Xd, ref
    api.reassign(X, ckv, w.iters, ws, w.seed)
    torch.cuda.synchronize()
    for h in (1, 40):
        _check_reassign_sample(X, ckv, h, w.T, 2000, seed=100 + h)


def test_stream_full_width_first_chunks():
    """The streaming workload at full width (720 tensors of 4680-token chunks) into a cache
    of full capacity (60 chunks, 280800 slots, 60 centroid tables): three chunks, the
    first cold and the next two warm-started from the previous chunk's tables, then one
    chunked dequant over the filled slots.  Sampled tensors are checked chunk by chunk."""
    w = synth.workload("stream_30x12_60chunk")
    n_chunks_total = w.frames // w.chunk_frames
    L = w.chunk_frames * w.gh * w.gw
    H = w.H
    dev = torch.device("cuda")
    cache = api.allocate(H, n_chunks_total * L, w.C, w.T, w.bits, w.group,
                         n_tables=n_chunks_total, device=dev)
    ws = api.new_workspace(H, L, w.C, w.T, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sample = (0, 1, 361, H - 1)
    Xs = []
    n_run = 3
    for c in range(n_run):
        Xc = w.make(dev, f0=c * w.chunk_frames, nf=w.chunk_frames)
        warm = None if c == 0 else cache.centroids[:, c - 1]
        api.quantize(Xc, w.C, w.T, w.bits, w.group, w.iters if c == 0 else w.warm_iters,
                     w.seed, warm=warm, warm_stride=cache.centroids.stride(0), out=cache,
                     token_offset=c * L, table_index=c, workspace=ws, status=status)
        Xs.append(Xc[list(sample)].cpu())
        del Xc
    filled = n_run * L
    xhat = torch.empty((len(sample), filled, 128), dtype=torch.float32, device=dev)
    # reconstruct only the sampled tensors: a cache view of those tensors
    sub = api.CompressedKV(cache.codes[list(sample)], cache.scales[list(sample)],
                           cache.pi[list(sample)], cache.centroids[list(sample)],
                           w.C, w.T, w.bits, w.group)
    api.dequantize(sub, filled, torch.float32, chunk_len=L, out=xhat, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status %#x" % int(status.item())
    codes, scales, pi = _np(sub.codes), _np(sub.scales), _np(sub.pi)
    cent, x32 = _np(sub.centroids), _np(xhat)
    for c in range(n_run):
        sl = slice(c * L, (c + 1) * L)
        for k, h in enumerate(sample):
            Xd = oracle.decode_input(Xs[c][k:k + 1])[0]
            qc.forced_check(Xd, codes[k, sl], scales[k, sl], pi[k, :, sl], cent[k, c],
                            w.bits, w.group)
            qc.check_reconstruction(x32[k, sl], codes[k, sl], scales[k, sl], pi[k, :, sl],
                                    cent[k, c], w.bits, w.group)
        # a warm chunk against the oracle continuing from the GPU's previous tables
        if c > 0:
            k, h = 1, sample[1]
            Xd = oracle.decode_input(Xs[c][k:k + 1])
            ref = oracle.quantize(Xd, w.C, w.T, w.bits, w.group, w.warm_iters, w.seed,
                                  tensor_id_base=h, warm=cent[k:k + 1, c - 1])
            qc.check_oracle_run(Xd[0], pi[k, :, sl], cent[k, c], ref["pi"][0],
                                ref["centroids"][0], ref["J"][0])
