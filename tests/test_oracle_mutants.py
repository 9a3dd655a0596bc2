"""The pins have teeth: each plausible mistake planted in a copy of the oracle
(a swapped word, a dropped term, a wrong sign or index, a transposed operand,
a non-strict comparison) makes the pin suite fail.  Mutants are compiled from
a modified copy of the source on the CPU; the oracle itself is untouched."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "sdv_oracle.c")
HDR = os.path.join(ROOT, "oracle", "sdv_oracle.h")

# (name, text in the source, replacement, occurrences to replace (0 = all))
MUTANTS = [
    ("philox_hi_for_lo", "uint32_t y1 = lo1;", "uint32_t y1 = hi1;", 1),
    ("philox_key_bump_first_round", "if (round > 0) {", "if (round >= 0) {", 1),
    ("philox_weyl_constant", "#define PHILOX_WEYL1 0xBB67AE85u", "#define PHILOX_WEYL1 0xBB67AE86u", 1),
    ("uniform_23_bits", "(double)(word >> 8) * (1.0 / 16777216.0)",
     "(double)(word >> 9) * (1.0 / 8388608.0)", 1),
    ("uniform_wrong_word", "if (u) *u = sdvo_uniform24(out[0]);", "if (u) *u = sdvo_uniform24(out[2]);", 1),
    ("counter_b_j_swapped", "uint32_t ctr[4] = {j, b, 0u, 0u};", "uint32_t ctr[4] = {b, j, 0u, 0u};", 1),
    ("lse_times_T", "double z = sdvo_logit(row, dtype, v) / T;", "double z = sdvo_logit(row, dtype, v) * T;", 0),
    ("lse_drops_max", "return m + log(s);", "return log(s);", 1),
    ("ratio_transposed", "return exp(lp - lq);", "return exp(lq - lp);", 1),
    ("ratio_q_zero_rejects", "if (lq == -INFINITY) return 1.0;", "if (lq == -INFINITY) return 0.0;", 1),
    ("streak_drops_product", "prefix *= a[j];", "prefix = a[j];", 1),
    ("streak_off_by_one", "prefix *= a[j];\n        score += prefix;",
     "score += prefix;\n        prefix *= a[j];", 1),
    ("argmax_last", "if (s[k] > s[best]) best = k;", "if (s[k] >= s[best]) best = k;", 1),
    ("accept_non_strict", "(u[j] < a[j])", "(u[j] <= a[j])", 1),
    ("cdf_non_strict", "if (c > t) {", "if (c >= t) {", 1),
    ("residual_transposed", "double d = pv - qv;", "double d = qv - pv;", 1),
    ("residual_unclipped", "r[v] = d > 0.0 ? d : 0.0;", "r[v] = d;", 1),
    ("bonus_wrong_uniform", "tok = sdvo_inverse_cdf(r, V, w[Lb], &R, &t, &c_prev, &c_v);",
     "tok = sdvo_inverse_cdf(r, V, w[0], &R, &t, &c_prev, &c_v);", 1),
    ("q_lse_from_p_row", "lse[i] = sdvo_row_lse(q_row(q_logits, sh, b, k, r - G - 1), dtype, V, T);",
     "lse[i] = sdvo_row_lse(p_row(p_logits, sh, b, k, r - G - 1), dtype, V, T);", 1),
    ("residual_drops_temperature", "double pv = exp(sdvo_logit(prow, dtype, v) / T - lse_p);",
     "double pv = exp(sdvo_logit(prow, dtype, v) - lse_p);", 1),
    ("greedy_ratio_squared", "    return exp(lp);                        /* accept with probability p(x)     */",
     "    return exp(2.0 * lp);", 1),
    ("greedy_keeps_rejected_token", "r[v] = v == xr ? 0.0 : exp(sdvo_logit(prow, dtype, v) / T - lse_p);",
     "r[v] = exp(sdvo_logit(prow, dtype, v) / T - lse_p);", 1),
    ("greedy_zeroes_wrong_token", "const int32_t xr = drafts[((int64_t)b * K + sel) * G + L];",
     "const int32_t xr = drafts[((int64_t)b * K + sel) * G + (L + 1) % G];", 1),
    ("cps_ties_to_higher_id", "return x->v < y->v ? -1 : (x->v > y->v ? 1 : 0);",
     "return x->v > y->v ? -1 : (x->v < y->v ? 1 : 0);", 1),
    ("cps_prune_ignores_temperature", "e[v].z = sdvo_logit(row, dtype, v) / T;",
     "e[v].z = sdvo_logit(row, dtype, v);", 1),
    ("cps_eos_dropped", "            Lc = j + 1;", "            Lc = j;", 1),
    ("cps_key_not_accumulated", "double key = cur[w].key + rl[j * mmax + r];",
     "double key = rl[j * mmax + r];", 1),
    ("cps_score_not_accumulated", "nxt[pos].score = cur[w].score + cl[j * mmax + r];",
     "nxt[pos].score = cl[j * mmax + r];", 1),
    ("cps_beam_one_short", "if (pos >= W) continue;", "if (pos >= (W > 1 ? W - 1 : 1)) continue;", 1),
    ("cps_ties_lexicographic_last", "        if (ra[i] < rb[i]) return 1;\n        if (ra[i] > rb[i]) return 0;",
     "        if (ra[i] > rb[i]) return 1;\n        if (ra[i] < rb[i]) return 0;", 1),
    ("cps_keeps_zero_probability", "        if (e[n].z == -INFINITY) break;", "", 1),
    ("len_scan_one_short", "int L = sdvo_accept_length(as, u, Lb);",
     "int L = sdvo_accept_length(as, u, Lb > 0 ? Lb - 1 : 0);", 1),
    ("len_bonus_uniform_of_gamma", "tok = sdvo_inverse_cdf(r, V, w[Lb], &R, &t, &c_prev, &c_v);",
     "tok = sdvo_inverse_cdf(r, V, w[G], &R, &t, &c_prev, &c_v);", 1),
    ("len_streak_over_gamma", "S[k] = sdvo_streak_score(a + (size_t)k * G, Lb);",
     "S[k] = sdvo_streak_score(a + (size_t)k * G, G);", 1),
    ("len_reads_past_length", "        if (r <= Lb)\n", "        if (r <= G)\n", 1),
    ("adl_pace_strict", "int keeps_pace = sa >= sg;", "int keeps_pace = sa > sg;", 1),
    ("adl_ignores_saturation", "int fills = sg >= sk;", "int fills = 1;", 1),
    ("adl_no_clamp_of_generated", "        if (g > kb) g = kb;", "", 1),
    ("adl_saturation_shrinks", "            next = kb;                /* generation saturated: hold */",
     "            next = kb - down;", 1),
    ("adl_window_one_short", "int n = seen < W ? (int)seen : W;", "int n = seen < W ? (int)seen : W - 1;", 1),
    ("adl_no_clamp_of_accepted", "        if (a > g) a = g;", "", 1),
]


@pytest.mark.slow
@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, count, tmp_path):
    src = open(SRC).read()
    assert old in src, "mutant %s no longer matches the source" % name
    mutated = src.replace(old, new) if count == 0 else src.replace(old, new, count)
    c = tmp_path / "sdv_oracle.c"
    c.write_text(mutated)
    (tmp_path / "sdv_oracle.h").write_text(open(HDR).read())
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", str(lib),
                    str(c), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, SDV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_greedy_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_cps_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_adl_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_len_pins.py")],
                       env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-1500:])
