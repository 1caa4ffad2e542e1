"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (derived from the arithmetic; see the design notes for the derivations):
  * codes and E4M3 scales, given the same assignments and centroids: bit-exact, except
    groups whose exact scale max|r|/qmax lies within 2^-20 (relative) of an E4M3 rounding
    midpoint and elements whose exact r/s_q lies within 2^-20 (relative) of a half-integer
    (of an integer for the mid-rise grid, whose codes change there).
    The GPU forms r as the fp32 value nearest the exact residual and divides in IEEE fp32,
    so it can only differ from the fp64 oracle inside those bands.  Band cases are counted.
  * centroids, given the same assignments: the fp32 rounding of the exact mean of the
    exact stage input, except within the compensated sum's error bound of a rounding
    midpoint (check_centroids gives the band); always within one fp32 ulp of the exact
    mean.  The GPU adds each residual as its fp32 value plus the rounding error of the
    chain that formed it, with TwoSum-compensated fp32 accumulation (about twice fp32's
    precision), and rounds the mean once.
  * reconstruction into fp32: |x_gpu - x_oracle| <= max(1e-3 * s_q, (T + 1) * ulp32(S)) with
    S = |deQ| + sum_t |C^(t)[pi^(t)]|: the GPU adds T + 1 fp32 terms in sequence, each add
    rounding by at most half an ulp of a partial sum bounded by S.
  * assignments from two independent runs: >= 99.9 % agreement per stage; the Lloyd
    objective within 1e-3 relative.
"""
from __future__ import annotations

import numpy as np

import oracle


def ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float64)).astype(np.float32)
    return np.spacing(np.maximum(x, np.float32(np.finfo(np.float32).tiny))).astype(np.float64)


def unpack_codes(codes, bits):
    codes = np.asarray(codes, dtype=np.uint8)
    per = 8 // bits
    mask = (1 << bits) - 1
    u = np.stack([(codes >> (bits * k)) & mask for k in range(per)], axis=-1)
    return u.reshape(*codes.shape[:-1], codes.shape[-1] * per).astype(np.int64)


def compare_codes(R, codes_gpu, scales_gpu, bits, group, eps=2.0 ** -20, scheme=0):
    """R: exact final residual [N][d] (fp64).  Returns counts; raises on a real mismatch.
    scheme 0: symmetric grid (codes change at half-integers of r/s_q); scheme 1: mid-rise
    (codes change at integers)."""
    qmax = (1 << (bits - 1)) - 1
    top = (1 << (bits - 1)) - 0.5 if scheme == 1 else qmax
    N, d = R.shape
    ng = d // group
    codes_o, scales_o = oracle.encode(R, bits, group, scheme)
    a = np.abs(R.reshape(N, ng, group)).max(axis=2)
    s = a / top
    sb_lo = oracle.e4m3_encode(s * (1 - eps))
    sb_hi = oracle.e4m3_encode(s * (1 + eps))
    band_group = sb_lo != sb_hi
    sq = oracle.e4m3_decode(scales_o)
    with np.errstate(divide="ignore", invalid="ignore"):
        # groups with s_q == 0 give inf / nan here; np.where below leaves them out
        v = R / np.repeat(sq, group, axis=1)
        if scheme == 1:
            frac = np.abs(v - np.rint(v))
        else:
            frac = np.abs(np.abs(v - np.floor(v)) - 0.5)
        band_elem = np.where(np.repeat(sq, group, axis=1) > 0,
                             frac <= eps * np.maximum(np.abs(v), 1.0), False)
    band_elem |= np.repeat(band_group, group, axis=1)
    scales_gpu = np.asarray(scales_gpu)
    bad_scales = (scales_gpu != scales_o) & ~band_group
    u_o = unpack_codes(codes_o, bits)
    u_g = unpack_codes(codes_gpu, bits)
    bad_codes = (u_o != u_g) & ~band_elem
    res = {"band_groups": int(band_group.sum()), "band_elems": int(band_elem.sum()),
           "scale_mismatch": int(bad_scales.sum()), "code_mismatch": int(bad_codes.sum()),
           "groups": int(band_group.size), "elems": int(band_elem.size)}
    if res["scale_mismatch"] or res["code_mismatch"]:
        i, g = np.argwhere(bad_scales)[0] if res["scale_mismatch"] else np.argwhere(bad_codes)[0]
        raise AssertionError("code/scale mismatch outside the rounding band: %s; first at "
                             "token %d group/elem %d" % (res, i, g))
    return res


def cluster_means(R_in, pi_t, C):
    """Exact (fp64) means of R_in's rows over each non-empty cluster of pi_t, and for each
    the band within which the GPU's compensated sum may leave it on either side of a
    rounding midpoint.

    The GPU adds the exact stage input (from the second stage on, each residual as its fp32
    value plus the rounding error of the chain that formed it) with TwoSum compensation, in
    runs of at most 32 sorted positions whose pieces are then added in order, and divides
    once.  With n members in p <= n/32 + 2 pieces and u = 2^-24, the error of its mean is at
    most (2^-38 + p (32 + p) u^2) times the members' mean magnitude (the error terms of one
    piece are added in fp32, at most 32 of them; those of the pieces, p of them), plus
    2^-46 of the mean for the corrected division.  The fp64 reference sum here adds at most
    n 2^-53 of the mean magnitude.  Returns (nonempty mask, exact means, band)."""
    pi_t = np.asarray(pi_t, dtype=np.int64)
    counts = np.bincount(pi_t, minlength=C)
    sums = np.zeros((C, R_in.shape[1]))
    np.add.at(sums, pi_t, R_in)
    sabs = np.zeros((C, R_in.shape[1]))
    np.add.at(sabs, pi_t, np.abs(R_in))
    nz = counts > 0
    n = counts[nz, None].astype(np.float64)
    exact = sums[nz] / n
    pieces = np.floor(n / 32.0) + 2.0
    band = (sabs[nz] / n) * (2.0 ** -38 + pieces * (32.0 + pieces) * 2.0 ** -48 + n * 2.0 ** -53) \
        + 2.0 ** -46 * np.abs(exact)
    return nz, exact, band


def check_centroids(R_in, pi_t, cent_gpu, stage):
    """fp32 centroids of one stage against the exact means of R_in over pi_t: the fp32
    rounding of the exact mean, except where it lies within the band of cluster_means of an
    fp32 rounding midpoint; everywhere within one fp32 ulp of the exact mean."""
    C = cent_gpu.shape[0]
    nz, exact, band = cluster_means(R_in, pi_t, C)
    got = cent_gpu[nz]
    err = np.abs(got.astype(np.float64) - exact)
    tol = ulp32(exact) + 1e-300
    worst = float((err / tol).max()) if err.size else 0.0
    if worst > 1.0:
        j = np.argwhere(err > tol)[0]
        raise AssertionError("stage %d centroid off by %.3g ulps (cluster row %d, channel %d)"
                             % (stage, worst, j[0], j[1]))
    want = exact.astype(np.float32)
    f = want.astype(np.float64)
    up = np.nextafter(want, np.float32(np.inf)).astype(np.float64)
    down = np.nextafter(want, np.float32(-np.inf)).astype(np.float64)
    near = (np.abs(exact - 0.5 * (f + up)) <= band) | (np.abs(exact - 0.5 * (f + down)) <= band)
    off = (got != want) & ~near
    if off.any():
        j, k = np.argwhere(off)[0]
        raise AssertionError("stage %d centroid (cluster row %d, channel %d) is %r, not the fp32 "
                             "rounding %r of the exact mean %r" % (stage, j, k, got[j, k],
                                                                  want[j, k], exact[j, k]))
    return {"clusters": int(nz.sum()), "empty": int((~nz).sum()), "worst_ulp_frac": worst,
            "exact_bits": int((got == want).sum()), "band": int(near.sum()),
            "entries": int(exact.size)}


def check_centroids_stored(R_in, pi_t, cent_gpu, stage, fmt):
    """Centroids of one stage in a 16-bit storage format (1 binary16, 2 bfloat16) against the
    oracle's rounding of the exact means of R_in over pi_t.  Each stored value must be
    representable in the format; a non-empty cluster's value must equal the rounding of its
    exact mean, except where the exact mean lies within the band of cluster_means of a
    midpoint of two format values (the GPU rounds a faithful fp32 mean and settles a mean
    exactly on a midpoint by the sign of what it leaves out, which is right outside that
    band).  There the value must be one of the two neighbours."""
    C = cent_gpu.shape[0]
    np.testing.assert_array_equal(oracle.store_centroids(cent_gpu.astype(np.float64), fmt),
                                  cent_gpu)
    nz, exact, band = cluster_means(R_in, pi_t, C)
    want = oracle.store_centroids(exact, fmt)
    lo = oracle.store_centroids(exact - band, fmt)
    hi = oracle.store_centroids(exact + band, fmt)
    got = cent_gpu[nz]
    differ = got != want
    ok = ~differ | ((lo != hi) & ((got == lo) | (got == hi)))
    if not ok.all():
        j, k = np.argwhere(~ok)[0]
        raise AssertionError("stage %d stored centroid (row %d, channel %d): got %r, want %r "
                             "(exact mean %r)" % (stage, j, k, got[j, k], want[j, k], exact[j, k]))
    return {"clusters": int(nz.sum()), "entries": int(exact.size),
            "tie_band": int(differ.sum())}


def forced_check(X, codes, scales, pi, cent, bits, group, scheme=0):
    """One tensor's GPU outputs against the oracle given the GPU's own assignments.
    X [N][d] fp64; pi [T][N]; cent [T][C][d]."""
    T = pi.shape[0]
    out = {"stages": []}
    R = np.array(X, dtype=np.float64)
    for t in range(T):
        out["stages"].append(check_centroids(R, pi[t], cent[t], t + 1))
        R = oracle.subtract(R, pi[t].astype(np.int32), cent[t])
    out["codes"] = compare_codes(R, codes, scales, bits, group, scheme=scheme)
    return out


def check_reconstruction(xhat_gpu, codes, scales, pi, cent, bits, group, scheme=0):
    """fp32 GPU reconstruction against the oracle's decode of the same compressed data."""
    T = pi.shape[0]
    want = oracle.dequantize(codes, scales, pi, cent, bits, group, scheme)
    deq = oracle.decode_codes(codes, scales, bits, group, scheme)
    S = np.abs(deq)
    for t in range(T):
        S = S + np.abs(cent[t][pi[t].astype(np.int64)])
    sq = np.repeat(oracle.e4m3_decode(scales), group, axis=1)
    tol = np.maximum(1e-3 * sq, (T + 1) * ulp32(S))
    err = np.abs(np.asarray(xhat_gpu, dtype=np.float64) - want)
    if not np.all(err <= tol):
        i, k = np.argwhere(err > tol)[0]
        raise AssertionError("reconstruction off at token %d channel %d: got %r want %r tol %r"
                             % (i, k, xhat_gpu[i, k], want[i, k], tol[i, k]))
    return {"max_err_over_tol": float((err / tol).max())}


def decode_with_slack(codes, scales, pi, cent, bits, group, scheme=0):
    """The oracle's fp64 reconstruction of one tensor and, per element, the most an fp32
    reconstruction can be off: (T + 1) * ulp32(|deQ| + sum_t |C^(t)[pi^(t)]|)."""
    T = pi.shape[0]
    x = oracle.dequantize(codes, scales, pi, cent, bits, group, scheme)
    S = np.abs(oracle.decode_codes(codes, scales, bits, group, scheme))
    for t in range(T):
        S = S + np.abs(cent[t][pi[t].astype(np.int64)])
    return x, (T + 1) * ulp32(S)


def attention_tolerance(Q, K, V, eps_k, eps_v, scale):
    """Bound on |O_fp32 - O_exact| per (query, channel) for attention computed in fp32 over
    keys and values rebuilt in fp32 (each off by at most eps_k / eps_v from K / V):
      * a score is a 128-term fp32 FMA chain times the scale:
        |ds| <= scale * (|q|.eps_k + 2 * 128 u * |q|.|k|) + 2u |s|   (u = 2^-24);
      * the softmax weights then move by a relative rho <= expm1(2 max|ds|) + 8u (two
        exponentials of 2 ulps and the rescaling products), which moves the weighted mean
        by at most 2 rho max|v| (the weights sum to one);
      * the sums of weights and weighted values (N terms, one rescale per 32-key tile, one
        per split when the splits are merged) add gamma = (N + N/16 + 4096) u relative to
        max|v| each, the final division one more u;
      * the values themselves are off by at most max eps_v."""
    u = 2.0 ** -24
    Q = np.asarray(Q, dtype=np.float64)
    N = K.shape[0]
    aq = np.abs(Q)
    ds = scale * (aq @ eps_k.T + 2 * 128 * u * (aq @ np.abs(K).T)) + 2 * u * np.abs(scale * (Q @ K.T))
    rho = np.expm1(2 * ds.max(axis=1)) + 8 * u
    gamma = (N + N / 16 + 4096) * u
    vmax = np.abs(V).max(axis=0)
    return (2 * rho[:, None] + 2 * gamma + u) * vmax[None, :] + eps_v.max(axis=0)[None, :] + 1e-30


def check_rounded_output(x16, x32, dtype):
    """A 16-bit output must be the round-to-nearest-even of the fp32 output."""
    import torch
    want = torch.from_numpy(np.asarray(x32, dtype=np.float32)).to(dtype)
    got = torch.as_tensor(x16).cpu()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def assignment_agreement(pi_gpu, pi_orc, R_stage_inputs, cent_orc):
    """Per stage: fraction of equal assignments and, for every mismatch, the relative
    distance gap against the oracle's centroids."""
    res = []
    for t in range(pi_gpu.shape[0]):
        eq = pi_gpu[t] == pi_orc[t]
        gaps = []
        R = R_stage_inputs[t]
        for i in np.flatnonzero(~eq):
            dg = ((R[i] - cent_orc[t][pi_gpu[t][i]]) ** 2).sum()
            do = ((R[i] - cent_orc[t][pi_orc[t][i]]) ** 2).sum()
            gaps.append((dg - do) / max(do, 1e-12 * (R[i] ** 2).sum(), 1e-300))
        res.append({"agree": float(eq.mean()), "mismatches": int((~eq).sum()),
                    "max_gap": float(max(gaps)) if gaps else 0.0})
    return res


def check_oracle_run(Xd, pi_gpu, cent_gpu, ref_pi, ref_cent, ref_J, min_agree=0.999,
                     max_gap=1e-3, j_rel=1e-3, stages=None):
    """One tensor's GPU run against the oracle's own independent run, stage by stage:
      * the assignments agree on at least `min_agree` of the tokens;
      * every token assigned differently is a near tie: its GPU cluster is at most `max_gap`
        farther (relative squared distance, on the oracle's stage input and centroids) than
        the oracle's;
      * the Lloyd objective J of the stage (the GPU's own assignment and centroids, on its
        own fp64 stage input) is within `j_rel` of the oracle's (plus 1e-12 of ||X||^2, for
        stages whose objective is zero).
    Xd [N][d] fp64; pi_* [T][N]; cent_* [T][C][d]; ref_J [T].  Returns the per-stage
    agreement records."""
    T = pi_gpu.shape[0] if stages is None else stages
    Rin = [oracle.residual(Xd, ref_pi, ref_cent, t) for t in range(T)]
    agr = assignment_agreement(pi_gpu[:T], ref_pi[:T], Rin, ref_cent)
    floor = 1e-12 * float((np.asarray(Xd, dtype=np.float64) ** 2).sum())
    for t, a in enumerate(agr):
        assert a["agree"] >= min_agree, ("stage", t + 1, a)
        assert a["max_gap"] <= max_gap, ("stage", t + 1, a)
        J = oracle.objective(oracle.residual(Xd, pi_gpu, cent_gpu, t),
                             np.asarray(pi_gpu[t], dtype=np.int32), cent_gpu[t])
        a["J_gpu"], a["J_oracle"] = J, float(ref_J[t])
        assert abs(J - ref_J[t]) <= j_rel * ref_J[t] + floor, ("stage", t + 1, a)
    return agr
