"""Planted mistakes in the oracle, on the CPU.

Each mutant is a copy of oracle/qvg_oracle.c with one plausible mistake: a flipped sign, a
dropped or extra term, a wrong index, constant or rounding rule.  The oracle's pins (the
CPU test files listed in PINS) run against every mutant through QVG_ORACLE_LIB and must
fail; an unmodified copy built the same way must pass.  A mutant that no pin catches is a
gap in the pins.  The attention oracle's mutants are numpy functions swapped in for it while
its pins run.  The mistakes are planted only in these copies, on the CPU.
"""
import concurrent.futures
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_pins.py", "tests/test_midrise_oracle.py",
        "tests/test_centroid_storage_oracle.py", "tests/test_attention_oracle.py"]

# (name, text in qvg_oracle.c, its replacement).  Every mutant keeps all memory accesses in
# bounds, so a mutant can only give wrong values, never crash the test process.
MUTANTS = [
    ("distance_sign", "double diff = r[k] - (double)c[k];", "double diff = r[k] + (double)c[k];"),
    ("distance_drops_last_channel", "for (int k = 0; k < d; k++) {\n        double diff",
     "for (int k = 0; k < d - 1; k++) {\n        double diff"),
    ("ties_to_highest", "if (D < best) {", "if (D <= best) {"),
    ("mean_divides_by_n_plus_1", "/ (double)n[j], format);", "/ (double)(n[j] + 1), format);"),
    ("mean_sums_wrong_channel", "sum[(int64_t)j * d + k] += R[i * d + k];",
     "sum[(int64_t)j * d + k] += R[i * d + (k + 1) % d];"),
    ("empty_cluster_zeroed", "if (n[j] == 0) continue;",
     "if (n[j] == 0) { for (int k = 0; k < d; k++) cent[(int64_t)j * d + k] = 0.f; continue; }"),
    ("subtract_adds", "R[i * d + k] -= (double)cent", "R[i * d + k] += (double)cent"),
    ("objective_keeps_last_term", "J += orc_sqdist(", "J = orc_sqdist("),
    ("scale_over_2_to_b_minus_1", "(double)mid - 0.5 : (double)qmax;",
     "(double)mid - 0.5 : (double)mid;"),
    ("rounds_half_away", "double q = nearbyint(r[k] / sq);", "double q = round(r[k] / sq);"),
    ("rounds_down", "double q = nearbyint(r[k] / sq);", "double q = floor(r[k] / sq);"),
    ("no_upper_clamp", "if (q > qmax) q = qmax;", ""),
    ("code_offset", "u = (int)q + mid;", "u = (int)q + mid - 1;"),
    ("absmax_drops_last_channel",
     "for (int k = g * group; k < (g + 1) * group; k++)\n                if (fabs(r[k]) > a)",
     "for (int k = g * group; k < (g + 1) * group - 1; k++)\n                if (fabs(r[k]) > a)"),
    ("decode_offset", "out[i * d + k] = sq * ((double)(u - mid) + off);",
     "out[i * d + k] = sq * ((double)(u - mid + 1) + off);"),
    ("midrise_nearest_instead_of_floor", "double f = floor(r[k] / sq) + mid;",
     "double f = nearbyint(r[k] / sq) + mid;"),
    ("midrise_no_half", "const double off = scheme == 1 ? 0.5 : 0.0;",
     "const double off = 0.0;"),
    ("dequant_skips_stage_1", "for (int t = T; t >= 1; t--) {", "for (int t = T; t >= 2; t--) {"),
    ("e4m3_bias", "v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 9);"),
    ("e4m3_subnormal_scale", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("e4m3_ties_to_odd", "(err == best_err && (c & 1) == 0 && (best & 1) == 1)",
     "(err == best_err && (c & 1) == 1 && (best & 1) == 0)"),
    ("e4m3_saturates_low", "if (a >= 448.0) return (uint8_t)(sign | 0x7E);",
     "if (a >= 448.0) return (uint8_t)(sign | 0x7D);"),
    ("splitmix_constant", "0xBF58476D1CE4E5B9ULL", "0xBF58476D1CE4E5B8ULL"),
    ("shuffle_drops_swap", "perm[k] = tmp;", "(void)tmp;"),
    ("binary16_precision", "orc_round_p(v, 11, -14, 65504.0)", "orc_round_p(v, 10, -14, 65504.0)"),
    ("binary16_emin", "orc_round_p(v, 11, -14, 65504.0)", "orc_round_p(v, 11, -15, 65504.0)"),
    ("bfloat16_emin", "orc_round_p(v, 8, -126, ldexp(255.0, 120))",
     "orc_round_p(v, 8, -125, ldexp(255.0, 120))"),
    ("store_ties_away", "double r = nearbyint(fabs(x) / q) * q;", "double r = round(fabs(x) / q) * q;"),
    ("stage_residual_not_updated", "orc_subtract(R, N, d, p, c); /* R^(t) */", "(void)0;"),
    ("warm_table_of_stage_1_for_all", "const float *w = warm + (int64_t)(t - 1) * C * d;",
     "const float *w = warm;"),
    ("cold_start_rows_of_x", "c[(int64_t)j * d + k] = orc_store(R[idx[j] * d + k],",
     "c[(int64_t)j * d + k] = orc_store(X[idx[j] * d + k],"),
    ("pi_of_every_stage_in_slot_1", "pi[(int64_t)(t - 1) * N + i] = (uint8_t)p[i];",
     "pi[i] = (uint8_t)p[i];"),
    ("encodes_x_not_the_residual", "orc_encode(R, N, d, cfg->bits", "orc_encode(X, N, d, cfg->bits"),
    ("packing_order_reversed", "(uint8_t)(u << ((k * bits) % 8));",
     "(uint8_t)(u << (8 - bits - (k * bits) % 8));"),
    ("e4m3_drops_sign", "return sign ? -v : v;", "return v;"),
    ("one_lloyd_round_short", "for (int it = 0; it < iters; it++) {",
     "for (int it = 1; it < iters; it++) {"),
    ("midrise_no_upper_clamp", "if (f > 2 * mid - 1) f = 2 * mid - 1;", ""),
    ("store_no_overflow", "if (r > maxfinite) r = INFINITY;", ""),
    ("tensor_id_ignored", "c, jb->tensor_id_base + h, jb->X", "c, jb->tensor_id_base, jb->X"),
]


def _build_and_run_pins(c_path: str, so: str) -> subprocess.CompletedProcess:
    oracle.compile_source(c_path, so)
    env = dict(os.environ, QVG_ORACLE_LIB=so)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           "-m", "not gpu", *PINS], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=900)


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    src = open(oracle._SRC).read()
    work = tmp_path_factory.mktemp("mutants")
    jobs = {}
    for name, old, new in [("unmodified", "", "")] + MUTANTS:
        if name != "unmodified":
            assert src.count(old) == 1, name
        c = work / (name + ".c")
        c.write_text(src.replace(old, new) if old else src)
        jobs[name] = (str(c), str(work / ("lib" + name + ".so")))
    workers = max(1, min(8, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        futs = {name: ex.submit(_build_and_run_pins, *job) for name, job in jobs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unmodified_copy_passes(results):
    r = results["unmodified"]
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_the_planted_mistake(results, name):
    r = results[name]
    # exit code 1: tests ran and one failed (not a crash, usage error or empty run)
    assert r.returncode == 1, "mutant %s: exit %d\n%s" % (name, r.returncode, r.stdout[-3000:])


# Planted mistakes in the attention oracle (numpy): each replaces oracle.attention.attention
# in this process while its pins run.
def _attn_no_shift(Q, K, V, scale):
    P = np.exp(float(scale) * (np.asarray(Q, float) @ np.asarray(K, float).T))
    return (P @ V) / P.sum(axis=1, keepdims=True)


def _attn_no_scale(Q, K, V, scale):
    S = np.asarray(Q, float) @ np.asarray(K, float).T
    P = np.exp(S - S.max(axis=1, keepdims=True))
    return (P @ V) / P.sum(axis=1, keepdims=True)


def _attn_keys_as_values(Q, K, V, scale):
    S = float(scale) * (np.asarray(Q, float) @ np.asarray(K, float).T)
    P = np.exp(S - S.max(axis=1, keepdims=True))
    return (P @ K) / P.sum(axis=1, keepdims=True)


def _attn_mean_not_weight_sum(Q, K, V, scale):
    S = float(scale) * (np.asarray(Q, float) @ np.asarray(K, float).T)
    P = np.exp(S - S.max(axis=1, keepdims=True))
    return (P @ V) / P.shape[1]


def _attn_shift_per_key(Q, K, V, scale):
    S = float(scale) * (np.asarray(Q, float) @ np.asarray(K, float).T)
    P = np.exp(S - S.max(axis=0, keepdims=True))
    return (P @ V) / P.sum(axis=1, keepdims=True)


ATTENTION_MUTANTS = [_attn_no_shift, _attn_no_scale, _attn_keys_as_values,
                     _attn_mean_not_weight_sum, _attn_shift_per_key]


@pytest.mark.parametrize("mutant", ATTENTION_MUTANTS, ids=lambda f: f.__name__[6:])
def test_attention_pins_catch_the_planted_mistake(monkeypatch, mutant):
    from oracle import attention as oatt
    from tests import test_attention_oracle as pins
    monkeypatch.setattr(oatt, "attention", mutant)
    runs = [(pins.test_matches_torch_sdpa_in_fp64, (M, N)) for M, N in ((1, 1), (3, 50), (16, 700))]
    runs += [(pins.test_one_key_gives_its_value, ()), (pins.test_equal_scores_give_the_mean_value, ()),
             (pins.test_a_leading_key_takes_all_the_weight, ()), (pins.test_invariances, ()),
             (pins.test_exact_cache_gives_attention_over_x, ())]
    failed = 0
    for fn, args in runs:
        try:
            with np.errstate(all="ignore"):
                fn(*args)
        except (AssertionError, ValueError, FloatingPointError):
            failed += 1
    assert failed > 0, mutant.__name__
