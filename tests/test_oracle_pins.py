"""Pins for the oracle: each test ties it to something other than itself.

Sources are the pages' worked example, closed forms, library routines (scipy's Lloyd,
torch's FP8 E4M3 cast), brute force on tiny inputs and invariants that follow from the
definitions.  Together they are chosen so that a dropped term, a wrong sign, a wrong index
or a transposed operand anywhere in the oracle fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    sections, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line[0].isalpha():
                cur = line
                sections[cur] = []
            else:
                sections[cur].append([float(v) for v in line.split()])
    return {k: np.array(v) for k, v in sections.items()}


def _ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float32))
    return np.spacing(np.maximum(x, np.float32(np.finfo(np.float32).tiny)))


# --------------------------------------------------------------------------------------
# Worked example from the pages
# --------------------------------------------------------------------------------------

def test_sky_example_centroid_is_group_mean():
    g = _read_golden("sky_vectors.txt")
    X = g["tokens"]
    want = g["centroid_numerators_over_3"][0] / 3.0
    cent, counts = oracle.update(X, np.zeros(3, np.int32), np.zeros((1, 4), np.float32))
    assert counts[0] == 3
    assert np.all(np.abs(cent[0] - want) <= _ulp32(want))
    # residuals of a group sum to zero up to the fp32 rounding of the stored centroid
    R = oracle.subtract(X, np.zeros(3, np.int32), cent)
    assert np.all(np.abs(R.sum(axis=0)) <= 3 * _ulp32(want))


# --------------------------------------------------------------------------------------
# FP8 E4M3 (OCP 8-bit floating point specification)
# --------------------------------------------------------------------------------------

def test_e4m3_spec_extremes():
    assert oracle.e4m3_decode([0x7E])[0] == 448.0          # largest finite
    assert oracle.e4m3_decode([0x08])[0] == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_decode([0x01])[0] == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_decode([0x07])[0] == 7 * 2.0 ** -9  # largest subnormal
    assert oracle.e4m3_decode([0x38])[0] == 1.0
    assert math.isnan(oracle.e4m3_decode([0x7F])[0])
    assert oracle.e4m3_decode([0xFE])[0] == -448.0
    assert oracle.e4m3_encode([1e6])[0] == 0x7E            # saturate to finite
    assert oracle.e4m3_encode([-1e30])[0] == 0xFE
    assert oracle.e4m3_encode([2.0 ** -11])[0] == 0x00     # below half the smallest step
    assert oracle.e4m3_encode([2.0 ** -10])[0] == 0x00     # exact tie -> even code 0
    assert oracle.e4m3_encode([3 * 2.0 ** -10])[0] == 0x02 # tie between codes 1 and 2 -> 2
    assert oracle.e4m3_encode([1.0625])[0] == 0x38         # tie 1.0 / 1.125 -> even (1.0)
    assert oracle.e4m3_encode([1.1875])[0] == 0x3A         # tie 1.125 / 1.25 -> even (1.25)


def test_e4m3_roundtrip_every_finite_code():
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = oracle.e4m3_decode(codes)
    assert np.all(np.diff(vals[:127]) > 0)  # monotone on the non-negative half
    back = oracle.e4m3_encode(vals)
    for c, b, v in zip(codes, back, vals):
        if c == 0x80:       # -0.0 keeps its sign bit
            assert b == 0x80
        else:
            assert b == c, (hex(c), v, hex(b))


def test_e4m3_matches_torch_cast():
    # torch's float8_e4m3fn cast (round to nearest even) as an independent library routine.
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(-448, 448, 20000),
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 20000)),
        # every midpoint between neighbouring codes, and a hair either side
        *[(lambda m: np.concatenate([m, np.nextafter(m, 0), np.nextafter(m, 1e9)]))(
            0.5 * (oracle.e4m3_decode(list(range(0, 0x7E))) +
                   oracle.e4m3_decode(list(range(1, 0x7F)))))],
    ]).astype(np.float32).astype(np.float64)
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------------------
# Seeded cold start
# --------------------------------------------------------------------------------------

def test_init_indices_distinct_in_range_and_seeded():
    a = oracle.init_indices(11, 3, 1, 1000, 256)
    assert len(set(a.tolist())) == 256 and a.min() >= 0 and a.max() < 1000
    assert np.array_equal(a, oracle.init_indices(11, 3, 1, 1000, 256))
    assert not np.array_equal(a, oracle.init_indices(11, 3, 2, 1000, 256))
    assert not np.array_equal(a, oracle.init_indices(11, 4, 1, 1000, 256))
    assert not np.array_equal(a, oracle.init_indices(12, 3, 1, 1000, 256))
    full = oracle.init_indices(5, 0, 1, 37, 37)
    assert sorted(full.tolist()) == list(range(37))


def test_splitmix_published_outputs_drive_the_shuffle():
    # SplitMix64 started from state 0 is published to emit 0xE220A8397B1DCDAF and then
    # 0x6E789E6AA1B965F4.  With seed 0, tensor id 0 and stage 0 the generator starts from
    # state 0, so the shuffle's first two picks follow from those two numbers.
    N = 1000003
    r1, r2 = 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4
    k1 = r1 % N
    k2 = 1 + r2 % (N - 1)
    idx = oracle.init_indices(0, 0, 0, N, 2)
    assert idx[0] == k1
    assert idx[1] == (0 if k2 == k1 else k2)


# --------------------------------------------------------------------------------------
# k-means (Lloyd) pins
# --------------------------------------------------------------------------------------

def _blobs(rng, n, d, k, spread=0.3, sep=5.0):
    centers = rng.standard_normal((k, d)) * sep
    lab = rng.integers(0, k, n)
    return centers[lab] + spread * rng.standard_normal((n, d)), lab


def test_lloyd_matches_scipy_kmeans2():
    from scipy.cluster.vq import kmeans2
    rng = np.random.default_rng(3)
    X, _ = _blobs(rng, 600, 16, 12, spread=1.0, sep=1.5)
    init = X[rng.choice(600, 12, replace=False)].astype(np.float32)
    for iters in (1, 3, 7):
        cent, pi = oracle.lloyd(X, init, iters)
        ref_c, ref_l = kmeans2(X, init.astype(np.float64), iter=iters, minit="matrix",
                               missing="warn")
        assert np.array_equal(pi, ref_l)
        assert np.allclose(cent, ref_c, rtol=1e-6, atol=1e-6)


def _all_two_partitions(n):
    for mask in range(1, 2 ** (n - 1)):
        lab = np.array([(mask >> i) & 1 for i in range(n)])
        yield lab


def test_exhaustive_two_means():
    rng = np.random.default_rng(5)
    for n in (4, 7, 10):
        X = rng.standard_normal((n, 3)) * np.array([3.0, 1.0, 0.5])
        best_J, best_lab = np.inf, None
        for lab in _all_two_partitions(n):
            J = sum(((X[lab == g] - X[lab == g].mean(0)) ** 2).sum() for g in (0, 1))
            if J < best_J:
                best_J, best_lab = J, lab
        # Lloyd from every pair of distinct points never beats the optimum
        for i, j in itertools.combinations(range(n), 2):
            cent, pi = oracle.lloyd(X, X[[i, j]].astype(np.float32), 20)
            assert oracle.objective(X, pi, cent) >= best_J * (1 - 1e-6)
        # started at the optimal centroids, Lloyd stays there
        opt_c = np.stack([X[best_lab == g].mean(0) for g in (0, 1)]).astype(np.float32)
        cent, pi = oracle.lloyd(X, opt_c, 5)
        assert np.array_equal(pi, best_lab)
        assert abs(oracle.objective(X, pi, cent) - best_J) <= 1e-5 * best_J


def test_objective_never_increases():
    rng = np.random.default_rng(9)
    X, _ = _blobs(rng, 500, 8, 20, spread=2.0, sep=1.0)
    cent = X[rng.choice(500, 20, replace=False)].astype(np.float32)
    prev = np.inf
    for _ in range(15):
        pi, _ = oracle.assign(X, cent)
        J_assign = oracle.objective(X, pi, cent)
        cent, _ = oracle.update(X, pi, cent)
        J_update = oracle.objective(X, pi, cent)
        assert J_assign <= prev * (1 + 1e-9)
        assert J_update <= J_assign * (1 + 1e-9)
        prev = J_update


def test_separated_mixture_is_recovered():
    rng = np.random.default_rng(1)
    X, lab = _blobs(rng, 400, 5, 4, spread=0.05, sep=10.0)
    # one init row from each true group
    init = np.stack([X[np.flatnonzero(lab == g)[0]] for g in range(4)]).astype(np.float32)
    cent, pi = oracle.lloyd(X, init, 5)
    assert np.array_equal(pi, lab)


def test_assignment_ties_go_to_lowest_index():
    X = np.array([[0.0, 0.0], [1.0, 0.0]])
    cent = np.array([[0.5, 1.0], [0.5, -1.0], [0.5, 1.0]], np.float32)
    pi, _ = oracle.assign(X, cent)
    assert pi.tolist() == [0, 0]


def test_empty_cluster_keeps_centroid():
    X = np.array([[0.0], [0.1], [0.2]])
    cent = np.array([[0.0], [100.0]], np.float32)
    new, counts = oracle.update(X, np.zeros(3, np.int32), cent)
    assert counts.tolist() == [3, 0] and new[1, 0] == 100.0


# --------------------------------------------------------------------------------------
# Whole path: special cases and invariants
# --------------------------------------------------------------------------------------

def _bf16_round(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().double().numpy()


def test_C_equals_N_gives_zero_residual_and_exact_reconstruction():
    rng = np.random.default_rng(2)
    X = _bf16_round(rng.standard_normal((1, 64, 128)) * 20)
    out = oracle.quantize(X, C=64, T=1, bits=2, group=32, iters=3, seed=4)
    assert sorted(out["pi"][0, 0].tolist()) == list(range(64))
    assert np.all(out["scales"] == 0)
    assert np.all(out["codes"] == 0b10101010)   # every code is the midpoint 2
    xh = oracle.dequantize(out["codes"][0], out["scales"][0], out["pi"][0],
                           out["centroids"][0], 2, 32)
    assert np.array_equal(xh, X[0])


def _rtn_reference(X, bits, group):
    """Textbook symmetric round-to-nearest group quantization with an E4M3 scale, written
    with numpy and torch's float8 cast, independent of the oracle."""
    qmax = 2 ** (bits - 1) - 1
    N, d = X.shape
    G = X.reshape(N, d // group, group)
    s = np.abs(G).max(axis=2) / qmax
    s8 = torch.from_numpy(np.minimum(s, 448.0).astype(np.float32)).to(torch.float8_e4m3fn)
    sq = s8.float().double().numpy()
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sq[..., None] > 0, np.clip(np.round(G / sq[..., None]), -qmax, qmax), 0)
    return s8.view(torch.uint8).numpy(), (q + 2 ** (bits - 1)).astype(np.int64).reshape(N, d), sq


@pytest.mark.parametrize("bits,group", [(2, 32), (2, 16), (4, 64), (4, 16)])
def test_T0_is_plain_group_rtn(bits, group):
    rng = np.random.default_rng(bits * 100 + group)
    # values chosen so that s = max/qmax is exactly an fp32 number away from E4M3 midpoints
    X = _bf16_round(rng.standard_normal((300, 128)) * np.where(rng.random(128) < 0.05, 50, 1))
    codes, scales = oracle.encode(X, bits, group)
    ref_s, ref_u, _ = _rtn_reference(X, bits, group)
    assert np.array_equal(scales, ref_s)
    per = 8 // bits
    unpacked = np.stack([(codes >> (bits * k)) & (2 ** bits - 1) for k in range(per)], axis=2)
    assert np.array_equal(unpacked.reshape(300, 128), ref_u)


@pytest.mark.parametrize("bits,group", [(2, 32), (4, 16)])
def test_T0_rtn_where_the_clamp_decides(bits, group):
    # Groups whose scale saturates at 448 (|r| in the thousands) and, at INT4, groups whose
    # scale falls among the subnormal E4M3 values and rounds down: there the nearest level
    # lies past qmax and the clamp decides the code.
    rng = np.random.default_rng(bits * 7 + group)
    mag = rng.choice([1e-2, 1.3e-2, 1.7e-2, 1.0, 2e3, 5e3], size=(400, 1))
    X = _bf16_round(rng.standard_normal((400, 128)) * mag)
    codes, scales = oracle.encode(X, bits, group)
    ref_s, ref_u, sq = _rtn_reference(X, bits, group)
    assert np.array_equal(scales, ref_s)
    per = 8 // bits
    unpacked = np.stack([(codes >> (bits * k)) & (2 ** bits - 1) for k in range(per)],
                        axis=2).reshape(400, 128)
    assert np.array_equal(unpacked, ref_u)
    qmax, mid = 2 ** (bits - 1) - 1, 2 ** (bits - 1)
    assert unpacked.min() >= mid - qmax and unpacked.max() <= mid + qmax
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.abs(X.reshape(400, 128 // group, group)) / sq[..., None]
    assert (ratio > qmax + 0.5).any()  # the case is exercised


def test_each_stage_starts_from_seeded_rows_of_its_input():
    # With one Lloyd round, a seeded row sits at distance ~0 (its fp32 rounding) from its own
    # starting centroid and far from the others, so it stays in that cluster: at every stage
    # pi^(t)[idx_j] = j, where idx are the stage's seeded indices and the starting centroids
    # are those rows of the stage input R^(t-1).
    rng = np.random.default_rng(12)
    X = _bf16_round(rng.standard_normal((1, 600, 128)) * 2 + rng.standard_normal(128) * 5)
    C, T, seed = 24, 3, 77
    ref = oracle.quantize(X, C, T, 2, 32, 1, seed)
    for t in range(1, T + 1):
        idx = oracle.init_indices(seed, 0, t, 600, C)
        assert np.array_equal(ref["pi"][0][t - 1][idx], np.arange(C)), t


def test_batch_equals_independent_tensors():
    # tensors of a batch are independent problems: tensor h of a batch is the single-tensor
    # call with tensor id h (its own seeded start), whatever else shares the batch
    rng = np.random.default_rng(13)
    X = _bf16_round(rng.standard_normal((3, 300, 128)) * 2 + rng.standard_normal((3, 1, 128)))
    ref = oracle.quantize(X, 16, 2, 2, 32, 2, 5)
    for h in range(3):
        one = oracle.quantize(X[h:h + 1], 16, 2, 2, 32, 2, 5, tensor_id_base=h)
        for k in ("codes", "scales", "pi", "centroids"):
            assert np.array_equal(ref[k][h], one[k][0]), (h, k)
    # and the seeded starts differ between tensor ids
    assert not np.array_equal(oracle.init_indices(5, 0, 1, 300, 16),
                              oracle.init_indices(5, 1, 1, 300, 16))


def test_code_packing_layout():
    # one token, d=16, INT2, group 16: values on the grid of scale 1.0 (E4M3 0x38)
    r = np.array([[1, 0, -1, 1, 0, 0, 1, -1, -1, -1, 0, 1, 1, 1, 1, 0]], np.float64)
    codes, scales = oracle.encode(r, 2, 16)
    assert scales.tolist() == [[0x38]]
    u = (r[0] + 2).astype(int)
    want = [u[0] | u[1] << 2 | u[2] << 4 | u[3] << 6, u[4] | u[5] << 2 | u[6] << 4 | u[7] << 6,
            u[8] | u[9] << 2 | u[10] << 4 | u[11] << 6, u[12] | u[13] << 2 | u[14] << 4 | u[15] << 6]
    assert codes[0].tolist() == want
    r4 = np.arange(-7, 9, dtype=np.float64)[None, :].clip(-7, 7)
    c4, s4 = oracle.encode(r4, 4, 16)
    assert s4.tolist() == [[0x38]]
    assert [(c4[0, k // 2] >> (4 * (k % 2))) & 15 for k in range(16)] == (r4[0] + 8).astype(int).tolist()


def test_grid_values_roundtrip_exactly():
    rng = np.random.default_rng(4)
    for bits in (2, 4):
        qmax = 2 ** (bits - 1) - 1
        sq = oracle.e4m3_decode(rng.integers(0x10, 0x60, (50, 4)).astype(np.uint8))
        q = rng.integers(-qmax, qmax + 1, (50, 4, 32))
        q[:, :, 0] = qmax  # the group maximum sits on the grid, so s = s_q exactly
        r = (q * sq[..., None]).reshape(50, 128)
        codes, scales = oracle.encode(r, bits, 32)
        assert np.array_equal(oracle.decode_codes(codes, scales, bits, 32), r)


def test_quantization_error_bound():
    rng = np.random.default_rng(8)
    R = rng.standard_normal((200, 128)) * np.exp(rng.uniform(-3, 3, (200, 1)))
    for bits, group in ((2, 32), (4, 16)):
        codes, scales = oracle.encode(R, bits, group)
        sq = np.repeat(oracle.e4m3_decode(scales), group, axis=1)
        err = np.abs(oracle.decode_codes(codes, scales, bits, group) - R)
        qmax = 2 ** (bits - 1) - 1
        inside = np.abs(R) <= qmax * sq
        assert np.all(err[inside] <= sq[inside] / 2 * (1 + 1e-12))
        assert np.all(err[~inside] <= np.abs(R[~inside]) - qmax * sq[~inside] + 1e-12)


def test_reconstruction_identity_and_residual_invariants():
    rng = np.random.default_rng(6)
    X = _bf16_round(rng.standard_normal((1, 700, 128)) * 3 + rng.standard_normal(128) * 10)
    T, C = 3, 16
    out = oracle.quantize(X, C=C, T=T, bits=2, group=32, iters=6, seed=9)
    pi, cent = out["pi"][0], out["centroids"][0]
    RT = oracle.residual(X[0], pi, cent, T)
    deq = oracle.decode_codes(out["codes"][0], out["scales"][0], 2, 32)
    xh = oracle.dequantize(out["codes"][0], out["scales"][0], pi, cent, 2, 32)
    # x - x_hat is exactly the quantization error of the final residual
    assert np.allclose(X[0] - xh, RT - deq, rtol=0, atol=1e-9)
    # codes are the encoding of the final residual
    codes, scales = oracle.encode(RT, 2, 32)
    assert np.array_equal(codes, out["codes"][0]) and np.array_equal(scales, out["scales"][0])
    # every stage's centroids are the means of its residual input over its assignment
    for t in range(T):
        Rin = oracle.residual(X[0], pi, cent, t)
        means, counts = oracle.update(Rin, pi[t].astype(np.int32), cent[t])
        assert np.array_equal(means, cent[t])
        Rout = oracle.subtract(Rin, pi[t].astype(np.int32), cent[t])
        for j in np.flatnonzero(counts):
            s = Rout[pi[t] == j].sum(axis=0)
            assert np.all(np.abs(s) <= counts[j] * _ulp32(cent[t][j]))
        assert np.isclose(out["J"][0, t], (Rout ** 2).sum(), rtol=1e-12)
    # the first stage removes the per-channel mean (no cluster is empty here)
    R1 = oracle.residual(X[0], pi, cent, 1)
    assert np.all(np.abs(R1.mean(axis=0)) <= np.abs(cent[0]).max() * 2e-7)


def test_warm_start_uses_the_given_centroids():
    rng = np.random.default_rng(10)
    X = _bf16_round(rng.standard_normal((2, 300, 128)))
    cold = oracle.quantize(X, C=8, T=2, bits=2, group=32, iters=4, seed=1)
    warm = oracle.quantize(X, C=8, T=2, bits=2, group=32, iters=4, seed=999,
                           warm=cold["centroids"])
    # Lloyd started from its own converged answer: one more round of 4 leaves a fixed point
    # whose objective is no worse
    assert np.all(warm["J"] <= cold["J"] * (1 + 1e-9))
    # and 0 iterations are not allowed: iters >= 1 always re-assigns
    with pytest.raises(ValueError):
        oracle.quantize(X, C=8, T=2, bits=2, group=32, iters=0, seed=1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_input_is_exact_over_every_16_bit_pattern(dtype):
    # the oracle reads the 16-bit inputs the GPU reads: every bit pattern decodes to the
    # value torch's own widening gives (NaNs stay NaN, signed zeros keep their sign)
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    x = bits.view(dtype)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to quiet NaNs
        got = oracle.decode_input(x)
    want = x.double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_input_keeps_fp32_and_float64_values():
    x = torch.tensor([1.0, -2.5, 3.0e-39, 1.0e38], dtype=torch.float32)
    assert np.array_equal(oracle.decode_input(x), x.double().numpy())
    a = np.array([0.1, -7.25])
    assert np.array_equal(oracle.decode_input(a), a)
