"""GPU parity: libqvg (through its C ABI) against the fp64 oracle on seeded inputs.

Each test uses sizes the oracle finishes in seconds but that still span several 128-token
GEMM tiles and a ragged tail; the full-size workloads are checked on sampled tensors with
properties that hold at any size.
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


def _to_np(ckv):
    return {k: getattr(ckv, k).cpu().numpy() for k in ("codes", "scales", "pi", "centroids")}


def _make(seed, H, frames, gh, gw, dtype=torch.bfloat16):
    tids = list(range(H))
    return synth.kv_tensor(seed, tids, 0, frames, gh, gw, dtype, "cpu")


def _gpu_quantize(X, C, T, bits, group, iters, seed, warm=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ckv = api.quantize(X.cuda(), C, T, bits, group, iters, seed,
                       warm=None if warm is None else torch.as_tensor(warm).cuda(),
                       status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status %#x" % int(status.item())
    return ckv


# --------------------------------------------------------------------------------------
# Fused dequant on the oracle's own compressed output
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("bits,group,T,C", [(2, 32, 2, 32), (4, 16, 1, 20), (2, 64, 3, 7),
                                            (4, 64, 0, 1), (2, 16, 4, 50)])
def test_dequant_matches_oracle(bits, group, T, C):
    X = _make(21, 3, 2, 17, 30)  # N = 1020: 7 full tiles and a ragged tail
    Xd = oracle.decode_input(X)
    ref = oracle.quantize(Xd, C, T, bits, group, 3, seed=5)
    H, N = X.shape[:2]
    ckv = api.allocate(H, N, C, T, bits, group, device="cuda")
    ckv.codes.copy_(torch.from_numpy(ref["codes"]))
    ckv.scales.copy_(torch.from_numpy(ref["scales"]))
    if T > 0:
        ckv.pi.copy_(torch.from_numpy(ref["pi"]))
        ckv.centroids.copy_(torch.from_numpy(ref["centroids"][:, None]))
    x32 = api.dequantize(ckv, out_dtype=torch.float32).cpu().numpy()
    x16 = api.dequantize(ckv, out_dtype=torch.bfloat16)
    xh16 = api.dequantize(ckv, out_dtype=torch.float16)
    for h in range(H):
        qc.check_reconstruction(x32[h], ref["codes"][h], ref["scales"][h], ref["pi"][h],
                                ref["centroids"][h], bits, group)
    qc.check_rounded_output(x16, x32, torch.bfloat16)
    qc.check_rounded_output(xh16, x32, torch.float16)


# --------------------------------------------------------------------------------------
# Encoding alone (T = 0 is plain group quantization)
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("bits,group", [(2, 32), (2, 16), (4, 64), (4, 16)])
def test_encode_T0_matches_oracle(dtype, bits, group):
    X = _make(3, 2, 3, 11, 31, dtype)
    if dtype == torch.float16:
        X = X.clamp(-6e4, 6e4)
    ckv = _gpu_quantize(X, 1, 0, bits, group, 1, 0)
    Xd = oracle.decode_input(X)
    for h in range(X.shape[0]):
        qc.compare_codes(Xd[h], ckv.codes[h].cpu().numpy(), ckv.scales[h].cpu().numpy(),
                         bits, group)


def test_encode_scale_edge_cases():
    # groups that saturate the E4M3 range, underflow it, sit exactly on grid points and
    # on E4M3 rounding midpoints
    rng = np.random.default_rng(0)
    N = 300
    Xf = rng.standard_normal((1, N, 128)).astype(np.float32)
    Xf[0, 0] *= 1e4                       # s > 448: saturates
    Xf[0, 1] *= 1e-5                      # s below the smallest subnormal / 2: zero scale
    Xf[0, 2] = 0.0                        # all-zero rows
    mids = 0.5 * (oracle.e4m3_decode(np.arange(1, 0x7E)) + oracle.e4m3_decode(np.arange(2, 0x7F)))
    for r in range(3, 3 + 40):
        Xf[0, r, :] = rng.uniform(-1, 1, 128)
        Xf[0, r, 0] = mids[(r * 7) % len(mids)]  # |max| / qmax(=1) hits a midpoint
    X = torch.from_numpy(Xf)
    ckv = _gpu_quantize(X, 1, 0, 2, 32, 1, 0)
    res = qc.compare_codes(Xf[0].astype(np.float64), ckv.codes[0].cpu().numpy(),
                           ckv.scales[0].cpu().numpy(), 2, 32)
    assert res["band_groups"] >= 1
    assert ckv.scales[0, 0].max().item() == 0x7E
    assert (ckv.scales[0, 2] == 0).all() and (ckv.codes[0, 2] == 0b10101010).all()


# --------------------------------------------------------------------------------------
# Assignment (tensor-core GEMM + exact near-tie re-scoring) and the mean update
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 7, 16, 37, 64, 200, 256])
def test_one_round_from_given_centroids(C):
    X = _make(8, 2, 3, 20, 21)  # N = 1260
    Xd = oracle.decode_input(X)
    H, N = X.shape[:2]
    rng = np.random.default_rng(C)
    warm = np.stack([Xd[h][rng.choice(N, C, replace=False)] for h in range(H)])[:, None]
    warm = warm.astype(np.float32)
    ckv = _gpu_quantize(X, C, 1, 2, 32, 1, 0, warm=warm)
    out = _to_np(ckv)
    for h in range(H):
        pi_o, _ = oracle.assign(Xd[h], warm[h, 0])
        agree = (out["pi"][h, 0] == pi_o).mean()
        assert agree == 1.0, agree
        qc.check_centroids(Xd[h], out["pi"][h, 0], out["centroids"][h, 0, 0], 1)


def test_assignment_with_outlier_channels_values():
    # value tensors: |x| up to 1e3 in four channels, the hardest case for the GEMM split
    X = synth.kv_tensor(4, [1, 3], 0, 2, 24, 40, torch.bfloat16, "cpu")  # odd ids = V
    Xd = oracle.decode_input(X)
    rng = np.random.default_rng(1)
    C = 128
    warm = np.stack([Xd[h][rng.choice(X.shape[1], C, replace=False)] for h in range(2)])
    warm = warm[:, None].astype(np.float32)
    ckv = _gpu_quantize(X, C, 1, 2, 32, 1, 0, warm=warm)
    pi = ckv.pi.cpu().numpy()
    for h in range(2):
        pi_o, _ = oracle.assign(Xd[h], warm[h, 0])
        assert (pi[h, 0] == pi_o).all()


@pytest.mark.parametrize("T,C", [(1, 256), (2, 256), (3, 48)])
def test_reassign_is_the_argmin_against_stored_centroids(T, C):
    X = _make(40 + T, 2, 3, 24, 36)  # N = 2592
    Xd = oracle.decode_input(X)
    H, N = X.shape[:2]
    ws = api.new_workspace(H, N, C, T)
    Xc = X.cuda()
    ckv = api.quantize(Xc, C, T, 2, 32, 3, 5, workspace=ws)
    api.reassign(Xc, ckv, 3, ws, 5)
    torch.cuda.synchronize()
    g = _to_np(ckv)
    for h in range(H):
        R = oracle.residual(Xd[h], g["pi"][h], g["centroids"][h, 0], T - 1)
        pi_o, _ = oracle.assign(R, g["centroids"][h, 0, T - 1])
        assert (g["pi"][h, T - 1] == pi_o).mean() >= 0.9999
    # the same steps one call at a time (qvg_reassign_steps) give the same bytes
    ckv.pi[:, T - 1].fill_(255)
    for step in (qvg.QVG_STEP_PLANES, qvg.QVG_STEP_GEMM, qvg.QVG_STEP_REFINE):
        api.reassign(Xc, ckv, 3, ws, 5, steps=step)
    torch.cuda.synchronize()
    assert np.array_equal(ckv.pi.cpu().numpy(), g["pi"])


def test_cold_start_indices_match_oracle():
    # with C = N every row is its own cluster, so pi reveals the seeded permutation
    N = 200
    X = _make(2, 3, 1, 10, 20)
    ckv = _gpu_quantize(X, N, 1, 2, 32, 1, seed=77)
    pi = ckv.pi.cpu().numpy()
    for h in range(3):
        idx = oracle.init_indices(77, h, 1, N, N)
        assert np.array_equal(pi[h, 0][idx], np.arange(N))
    assert (ckv.scales == 0).all()  # zero residual everywhere


# --------------------------------------------------------------------------------------
# Whole path against the oracle
# --------------------------------------------------------------------------------------

CASES = [
    # H, frames, gh, gw, C, T, bits, group, iters, dtype
    (2, 2, 17, 30, 16, 1, 2, 32, 4, torch.bfloat16),
    (2, 3, 20, 50, 64, 2, 2, 32, 5, torch.bfloat16),
    (2, 2, 23, 29, 37, 3, 4, 16, 3, torch.float16),
    (1, 2, 16, 40, 100, 2, 2, 64, 3, torch.float32),
    (2, 1, 9, 13, 5, 2, 4, 64, 6, torch.bfloat16),      # N = 117 < one tile
]


@pytest.mark.parametrize("case", CASES)
def test_end_to_end_matches_oracle(case):
    H, fr, gh, gw, C, T, bits, group, iters, dtype = case
    X = _make(100 + C, H, fr, gh, gw, dtype)
    Xd = oracle.decode_input(X)
    ckv = _gpu_quantize(X, C, T, bits, group, iters, seed=9)
    g = _to_np(ckv)
    ref = oracle.quantize(Xd, C, T, bits, group, iters, seed=9)
    x32 = api.dequantize(ckv, out_dtype=torch.float32).cpu().numpy()
    for h in range(H):
        qc.forced_check(Xd[h], g["codes"][h], g["scales"][h], g["pi"][h], g["centroids"][h, 0],
                        bits, group)
        qc.check_reconstruction(x32[h], g["codes"][h], g["scales"][h], g["pi"][h],
                                g["centroids"][h, 0], bits, group)
        qc.check_oracle_run(Xd[h], g["pi"][h], g["centroids"][h, 0], ref["pi"][h],
                            ref["centroids"][h], ref["J"][h])


def test_single_head_workload_matches_oracle():
    w = synth.workload("single_head_4x32x32")
    X = w.make()
    Xd = oracle.decode_input(X)
    ckv = _gpu_quantize(X, w.C, w.T, w.bits, w.group, w.iters, w.seed)
    g = _to_np(ckv)
    ref = oracle.quantize(Xd, w.C, w.T, w.bits, w.group, w.iters, w.seed)
    qc.check_oracle_run(Xd[0], g["pi"][0], g["centroids"][0, 0], ref["pi"][0],
                        ref["centroids"][0], ref["J"][0])
    qc.forced_check(Xd[0], g["codes"][0], g["scales"][0], g["pi"][0], g["centroids"][0, 0],
                    w.bits, w.group)
    x32 = api.dequantize(ckv, out_dtype=torch.float32).cpu().numpy()
    qc.check_reconstruction(x32[0], g["codes"][0], g["scales"][0], g["pi"][0],
                            g["centroids"][0, 0], w.bits, w.group)


def test_streaming_chunks_warm_start_and_chunked_dequant():
    # 4 chunks of 2 frames; chunk 0 cold, later chunks warm-started from the previous
    # chunk's table slot, written into one cache; then one dequant over all chunks
    H, fr, gh, gw, C, T, bits, group = 2, 2, 12, 20, 24, 2, 2, 32
    n_chunks, cold_iters, warm_iters = 4, 5, 2
    L = fr * gh * gw
    cache = api.allocate(H, n_chunks * L, C, T, bits, group, n_tables=n_chunks, device="cuda")
    ws = api.new_workspace(H, L, C, T)
    Xs = [synth.kv_tensor(31, [0, 1], c * fr, fr, gh, gw, torch.bfloat16, "cpu")
          for c in range(n_chunks)]
    for c in range(n_chunks):
        warm = None if c == 0 else cache.centroids[:, c - 1]
        api.quantize(Xs[c].cuda(), C, T, bits, group, cold_iters if c == 0 else warm_iters, 3,
                     warm=warm, warm_stride=cache.centroids.stride(0), out=cache,
                     token_offset=c * L, table_index=c, workspace=ws)
    x32 = api.dequantize(cache, out_dtype=torch.float32, chunk_len=L).cpu().numpy()
    g = _to_np(cache)
    warm_o = None
    for c in range(n_chunks):
        Xd = oracle.decode_input(Xs[c])
        ref = oracle.quantize(Xd, C, T, bits, group, cold_iters if c == 0 else warm_iters, 3,
                              warm=warm_o)
        sl = slice(c * L, (c + 1) * L)
        for h in range(H):
            qc.check_oracle_run(Xd[h], g["pi"][h, :, sl], g["centroids"][h, c], ref["pi"][h],
                                ref["centroids"][h], ref["J"][h])
            qc.forced_check(Xd[h], g["codes"][h, sl], g["scales"][h, sl], g["pi"][h, :, sl],
                            g["centroids"][h, c], bits, group)
            qc.check_reconstruction(x32[h, sl], g["codes"][h, sl], g["scales"][h, sl],
                                    g["pi"][h, :, sl], g["centroids"][h, c], bits, group)
        # the oracle continues from the GPU's tables, so each chunk is compared on its own
        warm_o = g["centroids"][:, c]


def test_repeat_runs_are_bitwise_identical():
    X = _make(5, 3, 2, 30, 30)
    a = _to_np(_gpu_quantize(X, 64, 2, 2, 32, 4, 1))
    b = _to_np(_gpu_quantize(X, 64, 2, 2, 32, 4, 1))
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_nonfinite_input_sets_status():
    X = _make(6, 1, 1, 16, 16)
    X[0, 17, 3] = float("nan")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.quantize(X.cuda(), 8, 1, 2, 32, 2, 0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & qvg.QVG_DEV_NONFINITE


def test_strided_input_and_token_offset():
    X = _make(12, 2, 2, 16, 16)  # N = 512
    big = torch.zeros((2, 700, 128), dtype=X.dtype)
    big[:, 100:612] = X
    view = big.cuda()[:, 100:612]
    cache = api.allocate(2, 1000, 16, 1, 2, 32, device="cuda")
    api.quantize(view, 16, 1, 2, 32, 3, 4, out=cache, token_offset=300)
    ref = _gpu_quantize(X, 16, 1, 2, 32, 3, 4)
    assert torch.equal(cache.codes[:, 300:812], ref.codes)
    assert torch.equal(cache.pi[:, :, 300:812], ref.pi)
    assert torch.equal(cache.centroids, ref.centroids)


def test_tensor_stride_off_the_row_grid_gives_the_same_bits():
    # A tensor stride that is not a whole number of 128-channel rows: the cluster sums
    # cannot address X as one [rows][128] view for their TMA row gathers and copy row by
    # row instead.  Both ways add the same values in the same order, so the results must
    # be the bits of the contiguous case.  T = 2 covers both stages' sums (the second one
    # also fetches the earlier stage's centroid rows).
    for dtype in (torch.bfloat16, torch.float32):
        X = _make(14, 3, 2, 18, 30, dtype)  # N = 1080
        H, N, _ = X.shape
        stride = N * 128 + 64  # 64 channels past a row boundary; 16-byte aligned
        flat = torch.zeros(H * stride, dtype=X.dtype, device="cuda")
        view = flat.as_strided((H, N, 128), (stride, 128, 1))
        view.copy_(X.cuda())
        args = (24, 2, 2, 32, 3, 6)
        got = _to_np(_gpu_quantize(view, *args))
        ref = _to_np(_gpu_quantize(X, *args))
        for k in ("codes", "scales", "pi", "centroids"):
            np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


@pytest.mark.parametrize("name", ["qvg", "qvg_pro"])
def test_presets_against_the_oracle(name):
    # The two named settings (one stage with 64-channel groups; four stages with 16-channel
    # groups) end to end against the oracle on a tensor pair of 4096 tokens: given the GPU's
    # assignments every stage's centroids, codes and scales are the oracle's (forced mode),
    # the reconstruction matches, and against the oracle's own Lloyd run every stage's
    # assignments agree on 99.9 % of tokens, every mismatch is a near tie and every stage's
    # objective is within 1e-3.
    from video_kv_cache_gb300.presets import PRESETS
    pr = PRESETS[name]
    X = _make(15, 2, 4, 32, 32)  # N = 4096
    iters, seed = 3, 11
    ckv = _gpu_quantize(X, pr.C, pr.T, pr.bits, pr.group, iters, seed)
    g = _to_np(ckv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x32 = api.dequantize(ckv, X.shape[1], torch.float32, status=status).cpu().numpy()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Xd = oracle.decode_input(X)
    ref = oracle.quantize(Xd, pr.C, pr.T, pr.bits, pr.group, iters, seed)
    for h in range(X.shape[0]):
        cent = g["centroids"][h, 0]
        qc.forced_check(Xd[h], g["codes"][h], g["scales"][h], g["pi"][h], cent, pr.bits, pr.group)
        qc.check_reconstruction(x32[h], g["codes"][h], g["scales"][h], g["pi"][h], cent,
                                pr.bits, pr.group)
        qc.check_oracle_run(Xd[h], g["pi"][h], cent, ref["pi"][h], ref["centroids"][h],
                            ref["J"][h])


# --------------------------------------------------------------------------------------
# The mid-rise grid (qscheme 1): 2^bits levels at half-integers of s_q
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("bits,group,T,C", [(2, 32, 2, 32), (4, 16, 1, 20), (2, 64, 0, 1),
                                            (4, 64, 3, 7)])
def test_midrise_dequant_matches_oracle(bits, group, T, C):
    # the fused dequant on the oracle's own mid-rise cache
    X = _make(22, 3, 2, 17, 30)  # N = 1020
    Xd = oracle.decode_input(X)
    ref = oracle.quantize(Xd, C, T, bits, group, 3, seed=5, scheme=1)
    H, N = X.shape[:2]
    ckv = api.allocate(H, N, C, T, bits, group, device="cuda")
    ckv.qscheme = qvg.QVG_QSCHEME_MIDRISE
    ckv.codes.copy_(torch.from_numpy(ref["codes"]))
    ckv.scales.copy_(torch.from_numpy(ref["scales"]))
    if T > 0:
        ckv.pi.copy_(torch.from_numpy(ref["pi"]))
        ckv.centroids.copy_(torch.from_numpy(ref["centroids"][:, None]))
    x32 = api.dequantize(ckv, out_dtype=torch.float32).cpu().numpy()
    x16 = api.dequantize(ckv, out_dtype=torch.bfloat16)
    for h in range(H):
        qc.check_reconstruction(x32[h], ref["codes"][h], ref["scales"][h], ref["pi"][h],
                                ref["centroids"][h], bits, group, scheme=1)
    qc.check_rounded_output(x16, x32, torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("bits,group", [(2, 32), (2, 16), (4, 64)])
def test_midrise_encode_T0_matches_oracle(dtype, bits, group):
    X = _make(4, 2, 3, 11, 31, dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ckv = api.quantize(X.cuda(), 1, 0, bits, group, 1, 0, status=status,
                       qscheme=qvg.QVG_QSCHEME_MIDRISE)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Xd = oracle.decode_input(X)
    for h in range(X.shape[0]):
        qc.compare_codes(Xd[h], ckv.codes[h].cpu().numpy(), ckv.scales[h].cpu().numpy(),
                         bits, group, scheme=1)


@pytest.mark.parametrize("bits,group,T", [(2, 32, 2), (4, 64, 1)])
def test_midrise_end_to_end(bits, group, T):
    X = _make(16, 2, 1, 24, 30)  # N = 720
    C, iters, seed = 32, 3, 9
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ckv = api.quantize(X.cuda(), C, T, bits, group, iters, seed, status=status,
                       qscheme=qvg.QVG_QSCHEME_MIDRISE)
    x32 = api.dequantize(ckv, X.shape[1], torch.float32, status=status).cpu().numpy()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = _to_np(ckv)
    Xd = oracle.decode_input(X)
    ref = oracle.quantize(Xd, C, T, bits, group, iters, seed, scheme=1)
    for h in range(X.shape[0]):
        cent = g["centroids"][h, 0]
        qc.forced_check(Xd[h], g["codes"][h], g["scales"][h], g["pi"][h], cent, bits, group,
                        scheme=1)
        qc.check_reconstruction(x32[h], g["codes"][h], g["scales"][h], g["pi"][h], cent, bits,
                                group, scheme=1)
        qc.check_oracle_run(Xd[h], g["pi"][h], cent, ref["pi"][h], ref["centroids"][h],
                            ref["J"][h])
        # the assignments do not depend on the grid: the symmetric run clusters the same way
        sym = oracle.quantize(Xd[h:h + 1], C, T, bits, group, iters, seed, tensor_id_base=h)
        np.testing.assert_array_equal(sym["pi"][0], ref["pi"][h])


def test_graph_capture_replays_identical_results():
    # qvg_quantize / qvg_dequantize enqueue only kernels and memsets on the given stream,
    # so a caller may capture them in a CUDA graph; the replay must give the same bits
    X = _make(13, 2, 2, 20, 30).cuda()
    H, N = X.shape[:2]
    C, T, bits, group, iters, seed = 32, 2, 2, 32, 3, 4
    out = api.allocate(H, N, C, T, bits, group, device="cuda")
    ws = api.new_workspace(H, N, C, T)
    xh = torch.empty((H, N, 128), dtype=torch.bfloat16, device="cuda")

    def step():
        api.quantize(X, C, T, bits, group, iters, seed, out=out, workspace=ws)
        api.dequantize(out, N, torch.bfloat16, out=xh)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = _to_np(out)
    ref_x = xh.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for k in ("codes", "scales", "pi", "centroids"):
        getattr(out, k).zero_()
    xh.zero_()
    g.replay()
    torch.cuda.synchronize()
    got = _to_np(out)
    for k in ref:
        assert np.array_equal(got[k], ref[k]), k
    assert torch.equal(xh, ref_x)
