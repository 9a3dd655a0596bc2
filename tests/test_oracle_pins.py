"""Pins of the fp64 CPU oracle against what the method and mathematics fix.

Nothing here re-types the oracle's own formulas: each check is a closed form,
an invariant, a published known-answer vector, a library routine for a special
case, an exact enumeration of the committed-token law, or a Monte-Carlo /
chi-square check of a probabilistic identity.

Passages: "SpecDiff-2: Scaling Diffusion Drafter Alignment For Faster
Speculative Decoding", section 2 (lossless acceptance rule, residual
replacement, distribution preserved), Figure 2 / section 3 (position-wise
acceptance and accepted streaks), section 5.2 (self-selection by a streak
score); "DiffuSpec: Unlocking Diffusion Language Models for Speculative
Decoding", section 3 (residual replacement is unbiased).
"""
import itertools
import os

import numpy as np
import pytest
from scipy import special, stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# Philox4x32-10
# ----------------------------------------------------------------------------

def test_philox_known_answer_vectors(oracle_lib):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        vals = [int(x, 16) for x in r]
        assert oracle_lib.philox4x32_10(vals[0:4], vals[4:6]) == vals[6:10]


def test_uniform24_range_and_keying(oracle_lib):
    assert oracle_lib.uniform24(0) == 0.0
    assert oracle_lib.uniform24(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle_lib.uniform24(0x000000FF) == 0.0          # low 8 bits dropped
    assert oracle_lib.uniform24(0x00000100) == 2.0 ** -24
    # counter (j, b, 0, 0), key (seed lo, seed hi); word 0 -> u, word 1 -> w
    seed, b, j = 0x0123456789ABCDEF, 7, 3
    words = oracle_lib.philox4x32_10([j, b, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
    u, w = oracle_lib.uniforms(seed, b, j)
    assert u == (words[0] >> 8) / 2.0 ** 24
    assert w == (words[1] >> 8) / 2.0 ** 24


def test_uniforms_are_uniform(oracle_lib):
    # Kolmogorov-Smirnov over 20k (b, j) pairs: the keyed stream is U[0,1).
    us, ws = [], []
    for b in range(2000):
        for j in range(10):
            u, w = oracle_lib.uniforms(42, b, j)
            us.append(u)
            ws.append(w)
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    assert stats.kstest(ws, "uniform").pvalue > 1e-3
    assert abs(np.corrcoef(us, ws)[0, 1]) < 0.03


# ----------------------------------------------------------------------------
# Temperature softmax (row LSE)
# ----------------------------------------------------------------------------

def _bf16_words(x):
    """Round float32 values to bf16 (nearest-even) and return raw words."""
    b = np.asarray(x, np.float32).view(np.uint32)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def test_lse_closed_forms(oracle_lib):
    for V in (1, 7, 32, 152064):
        for T in (0.6, 1.0, 2.5):
            row = np.full(V, 1.75, np.float32)
            assert oracle_lib.row_lse(row, T) == pytest.approx(1.75 / T + np.log(V), rel=1e-13)
    # two entries: LSE(a, b) = max + log(1 + exp(-|a - b|))
    for a, b, T in [(0.0, 0.0, 1.0), (3.0, -1.0, 0.7), (-20.0, 5.0, 1.3)]:
        za, zb = a / T, b / T
        expect = max(za, zb) + np.log1p(np.exp(-abs(za - zb)))
        assert oracle_lib.row_lse(np.array([a, b], np.float32), T) == pytest.approx(expect, rel=1e-14)


def test_lse_bf16_decoding(oracle_lib):
    # single-entry rows: LSE = l / T; bf16 words 0x3F80 = 1, 0xC000 = -2, 0x3FC0 = 1.5,
    # 0x4049 = 3.140625
    for word, value in [(0x3F80, 1.0), (0xC000, -2.0), (0x3FC0, 1.5), (0x4049, 3.140625)]:
        assert oracle_lib.row_lse(np.array([word], np.uint16), 0.5) == value / 0.5
    # -inf entries carry no mass; NaN / +inf rows and all -inf rows are flagged
    row = np.array([0x3F80, 0xFF80, 0x3F80], np.uint16)
    assert oracle_lib.row_lse(row, 1.0) == pytest.approx(1.0 + np.log(2.0), rel=1e-15)
    assert np.isnan(oracle_lib.row_lse(np.array([0x3F80, 0x7F80], np.uint16), 1.0))
    assert np.isnan(oracle_lib.row_lse(np.array([0x3F80, 0x7FC1], np.uint16), 1.0))
    assert oracle_lib.row_lse(np.array([0xFF80, 0xFF80], np.uint16), 1.0) == -np.inf


def test_lse_matches_library_logsumexp(oracle_lib):
    rng = np.random.default_rng(0)
    for V, T in [(32, 1.0), (1000, 0.7), (152064, 0.6)]:
        x = (rng.standard_normal(V) * 3 - 1.1 * np.log1p(np.arange(V))).astype(np.float32)
        words = _bf16_words(x)
        vals = (words.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert oracle_lib.row_lse(words, T) == pytest.approx(special.logsumexp(vals / T), rel=1e-13)
        assert oracle_lib.row_lse(x, T) == pytest.approx(
            special.logsumexp(x.astype(np.float64) / T), rel=1e-13)


def test_lse_shift_invariance(oracle_lib):
    rng = np.random.default_rng(1)
    # multiples of 2^-10 below 16 in magnitude: x + c is exact in float32
    x = (np.round(np.clip(rng.standard_normal(5000), -15, 15) * 1024) / 1024).astype(np.float32)
    for c in (1.0, -8.0, 64.0):
        assert oracle_lib.row_lse(x + np.float32(c), 0.8) == pytest.approx(
            oracle_lib.row_lse(x, 0.8) + c / 0.8, rel=1e-13)


# ----------------------------------------------------------------------------
# Acceptance ratio, streak, selection, acceptance scan, inverse CDF
# ----------------------------------------------------------------------------

def _softmax(l, T):
    return special.softmax(np.asarray(l, np.float64) / T)


def test_acceptance_probability_closed_form(oracle_lib):
    """E_{x~q}[min(1, p(x)/q(x))] = sum_v min(p_v, q_v)."""
    rng = np.random.default_rng(2)
    for V, T in [(2, 1.0), (8, 0.7), (32, 1.0), (500, 1.3)]:
        lp = (rng.standard_normal(V) * 2).astype(np.float32)
        lq = (lp + rng.standard_normal(V)).astype(np.float32)
        Lp, Lq = oracle_lib.row_lse(lp, T), oracle_lib.row_lse(lq, T)
        q = _softmax(lq, T)
        p = _softmax(lp, T)
        expect = np.minimum(p, q).sum()
        got = sum(q[x] * oracle_lib.accept_ratio(float(lp[x]) / T - Lp, float(lq[x]) / T - Lq)
                  for x in range(V))
        assert got == pytest.approx(expect, rel=1e-12)


def test_accept_ratio_conventions(oracle_lib):
    assert oracle_lib.accept_ratio(-1.0, -np.inf) == 1.0      # q(x) = 0
    assert oracle_lib.accept_ratio(-np.inf, -2.0) == 0.0      # p(x) = 0 < q(x)
    assert oracle_lib.accept_ratio(-1.0, -1.0) == 1.0         # q == p
    assert oracle_lib.accept_ratio(-0.5, -1.0) == 1.0         # q < p
    assert oracle_lib.accept_ratio(np.log(0.2), np.log(0.8)) == pytest.approx(0.25, rel=1e-15)


def test_streak_score_closed_forms(oracle_lib):
    assert oracle_lib.streak_score([1.0] * 16) == 16.0
    assert oracle_lib.streak_score([0.0, 1.0, 1.0]) == 0.0
    assert oracle_lib.streak_score([0.5] * 3) == 0.875          # 1/2 + 1/4 + 1/8
    r = 0.9                                                     # geometric sum
    assert oracle_lib.streak_score([r] * 20) == pytest.approx(r * (1 - r ** 20) / (1 - r), rel=1e-14)


def test_argmax_first_and_accept_length(oracle_lib):
    assert oracle_lib.argmax_first([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle_lib.argmax_first([5.0, 5.0]) == 0
    a = [1.0, 0.5, 0.2]
    assert oracle_lib.accept_length(a, [0.99, 0.4, 0.3]) == 2
    assert oracle_lib.accept_length(a, [0.99, 0.5, 0.1]) == 1   # u == a rejects (strict)
    assert oracle_lib.accept_length(a, [0.99, 0.1, 0.1]) == 3
    assert oracle_lib.accept_length([0.0], [0.0]) == 0


def test_inverse_cdf_intervals(oracle_lib):
    rng = np.random.default_rng(3)
    r = rng.random(12)
    r[[2, 5, 6]] = 0.0
    c = np.cumsum(r)
    R = c[-1]
    for v in range(12):
        lo = c[v - 1] if v else 0.0
        if r[v] == 0:
            continue
        for frac in (0.01, 0.5, 0.99):                          # interior of [C_{v-1}, C_v)
            w = (lo + frac * r[v]) / R
            assert oracle_lib.inverse_cdf(r, w)[0] == v
    for w in np.linspace(0, 1 - 2 ** -24, 4001):                # zero-mass ids never drawn
        assert r[oracle_lib.inverse_cdf(r, w)[0]] > 0
    # strict: t exactly on C_0 moves to the next id
    assert oracle_lib.inverse_cdf(np.ones(4), 0.25)[0] == 1
    assert oracle_lib.inverse_cdf(np.zeros(4), 0.5)[0] == -1


# ----------------------------------------------------------------------------
# Exact enumeration of the committed-token law (explicit uniforms placed at
# interval midpoints, each weighted by its interval's probability).
# ----------------------------------------------------------------------------

def _branches(p_rows, q_rows, drafts_k, T):
    """For one draft, the (L, weight, u vector, [(w, weight)]) branches of the
    acceptance scan and the final draw, from the test's own softmax."""
    G = len(drafts_k)
    a = []
    for j, x in enumerate(drafts_k):
        p, q = _softmax(p_rows[j], T), _softmax(q_rows[j], T)
        a.append(min(1.0, p[x] / q[x]))
    out = []
    prefix = 1.0
    for L in range(G + 1):
        if L < G:
            wt = prefix * (1.0 - a[L])
            u = [a[i] / 2 for i in range(L)] + [(1 + a[L]) / 2] + [0.5] * (G - L - 1)
            p, q = _softmax(p_rows[L], T), _softmax(q_rows[L], T)
            r = np.maximum(p - q, 0.0)
        else:
            wt = prefix
            u = [a[i] / 2 for i in range(G)]
            r = _softmax(p_rows[G], T)
        if L < G:
            prefix *= a[L]
        if wt <= 0:
            continue
        c = np.cumsum(r) / r.sum()
        draws = []
        for v in range(len(r)):
            if r[v] <= 0:
                continue
            lo = c[v - 1] if v else 0.0
            draws.append(((lo + c[v]) / 2, r[v] / r.sum(), v))
        out.append((L, wt, u, draws))
    return out


def _run_branches(oracle_lib, cases, T):
    """cases: list of (prob, p_logits [K,G+1,V], q_logits [K,G,V], drafts [K,G],
    u [G], w_index, w) -> oracle outputs for each, batched."""
    P = np.stack([c[1] for c in cases]).astype(np.float32)
    Q = np.stack([c[2] for c in cases]).astype(np.float32)
    D = np.stack([c[3] for c in cases]).astype(np.int32)
    G = D.shape[-1]
    U = np.array([c[4] for c in cases], np.float64).reshape(len(cases), G)
    W = np.full((len(cases), G + 1), 0.5)
    for i, c in enumerate(cases):
        W[i, c[5]] = c[6]
    return oracle_lib.verify_uniforms(P, Q, D, T, U, W)


def test_lossless_k1_exhaustive(oracle_lib):
    """K = 1: the committed token at every position, given that the step
    reaches it and the committed prefix, follows the verifier's conditional
    exactly (V <= 8, gamma <= 3; verifier conditionals depend on the prefix,
    drafter marginals on the position only, as in a one-pass diffusion draft)."""
    rng = np.random.default_rng(4)
    for V, G, T in [(3, 1, 1.0), (4, 2, 0.8), (3, 3, 1.0), (8, 2, 1.3)]:
        vrow = {}

        def verifier_row(prefix):
            if prefix not in vrow:
                vrow[prefix] = (rng.standard_normal(V) * 1.5).astype(np.float32)
            return vrow[prefix]

        q_rows = (rng.standard_normal((G, V)) * 1.5).astype(np.float32)
        qm = [_softmax(q_rows[j], T) for j in range(G)]
        cases, meta = [], []
        for x in itertools.product(range(V), repeat=G):
            px = np.prod([qm[j][x[j]] for j in range(G)])
            p_rows = np.stack([verifier_row(tuple(x[:j])) for j in range(G + 1)])
            for L, wt, u, draws in _branches(p_rows, q_rows, x, T):
                for wv, wwt, v in draws:
                    cases.append((px * wt * wwt, p_rows[None], q_rows[None],
                                  np.array(x)[None], u, L, wv))
                    meta.append((x, L, v))
        out = _run_branches(oracle_lib, cases, T)
        assert (out["sel"] == 0).all()
        assert (out["err"] == 0).all()
        law = {}
        for (x, L, v), c, ol, ot in zip(meta, cases, out["accept_len"], out["next_token"]):
            assert ol == L and ot == v          # the oracle's decision on each branch
            y = tuple(x[:L]) + (v,)
            law[y] = law.get(y, 0.0) + c[0]
        assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
        # P(y_{n+1} = v | at least n+1 committed, y_<=n) = p(v | y_<=n)
        for n in range(G + 1):
            prefixes = {y[:n] for y in law if len(y) > n}
            for pre in prefixes:
                mass = np.zeros(V)
                for y, m in law.items():
                    if len(y) > n and y[:n] == pre:
                        mass[y[n]] += m
                np.testing.assert_allclose(mass / mass.sum(), _softmax(verifier_row(pre), T),
                                           rtol=0, atol=1e-12)


def _first_token_law(oracle_lib, p_rows, q_rows, K, T, V):
    """Exact law of the first committed token with K drafts drawn i.i.d. from
    the drafter's marginals, by enumeration."""
    G = q_rows.shape[0]
    qm = [_softmax(q_rows[j], T) for j in range(G)]
    law = np.zeros(V)
    per_draft = list(itertools.product(range(V), repeat=G))
    cases = []
    for xs in itertools.product(per_draft, repeat=K):
        px = np.prod([qm[j][x[j]] for x in xs for j in range(G)])
        P = np.repeat(p_rows[None], K, 0)
        Q = np.repeat(q_rows[None], K, 0)
        D = np.array(xs)
        # the selected draft is decided before any uniform is used: find it
        sel = oracle_lib.verify_uniforms(P[None].astype(np.float32), Q[None].astype(np.float32),
                                         D[None], T, np.zeros((1, G)), np.zeros((1, G + 1)))["sel"][0]
        for L, wt, u, draws in _branches(p_rows, q_rows, xs[sel], T):
            for wv, wwt, v in draws:
                cases.append((px * wt * wwt, P, Q, D, u, L, wv))
    out = _run_branches(oracle_lib, cases, T)
    for i, c in enumerate(cases):
        s, L, tok = out["sel"][i], out["accept_len"][i], out["next_token"][i]
        y1 = c[3][s][0] if L > 0 else tok
        law[y1] += c[0]
    return law


def test_self_selection_counterexample_law(oracle_lib):
    """Golden: exact first-token law of the hand-derived K = 2 example; K = 1 is p."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "selfselect_counterexample.txt"))
            if l.strip() and not l.startswith("#")]
    p_rows = np.log(np.array([[0.5, 0.5], [0.5, 0.5]], np.float64)).astype(np.float32)
    q_rows = np.log(np.array([[0.9, 0.1]], np.float64)).astype(np.float32)
    for r in rows:
        K, expect = int(r[0]), np.array([float(r[1]), float(r[2])])
        law = _first_token_law(oracle_lib, p_rows, q_rows, K, 1.0, 2)
        np.testing.assert_allclose(law, expect, atol=1e-6)


def test_q_equals_p_invariant(oracle_lib):
    """q == p bitwise: every ratio is 1, every streak is gamma, draft 0 is
    selected, all gamma tokens are accepted and the bonus token follows p_gamma."""
    rng = np.random.default_rng(5)
    B, K, G, V = 64, 3, 5, 40
    P = _bf16_words(rng.standard_normal((B, K, G + 1, V)) * 3)
    Q = P[:, :, :G].copy()
    D = rng.integers(0, V, (B, K, G)).astype(np.int32)
    out = oracle_lib.verify(P, Q, D, 1.0, seed=9)
    assert (out["accept_len"] == G).all() and (out["sel"] == 0).all()
    assert (out["scores"] == G).all() and (out["ratio"] == 1.0).all()
    assert not (out["band"] & oracle_lib.BAND_SELECT).any()      # exact ties are not boundary
    # bonus token: exact inverse CDF of p_gamma at w_gamma, by interval
    for b in range(B):
        _, w = oracle_lib.uniforms(9, b, G)
        vals = (P[b, 0, G].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        c = np.cumsum(special.softmax(vals))
        assert out["next_token"][b] == int(np.searchsorted(c, w * c[-1], side="right"))


def test_expected_streak_equals_mean_accepted_length(oracle_lib):
    """E[L] over the acceptance uniforms = S (Monte Carlo, K = 1, fixed draft)."""
    rng = np.random.default_rng(6)
    G, V, N = 6, 16, 100_000
    p1 = (rng.standard_normal((G + 1, V)) * 1.0).astype(np.float32)
    q1 = (p1[:G] + rng.standard_normal((G, V)) * 0.8).astype(np.float32)
    x = np.array([int(np.argmax(q1[j])) for j in range(G)], np.int32)
    P = np.broadcast_to(p1, (N, 1, G + 1, V))
    Q = np.broadcast_to(q1, (N, 1, G, V))
    D = np.broadcast_to(x, (N, 1, G))
    out = oracle_lib.verify(P, Q, D, 1.0, seed=11, nthreads=oracle_lib.max_threads())
    S = out["scores"][0, 0]
    L = out["accept_len"].astype(np.float64)
    assert 0.5 < S < G - 0.5
    assert abs(L.mean() - S) < 5 * L.std() / np.sqrt(N)


@pytest.mark.slow
def test_chi_square_first_token_follows_verifier(oracle_lib):
    """10^6 seeded K = 1 trials on tiny-exact-style inputs (V = 32, gamma = 4,
    fp32, l_p ~ N(0, 2^2), l_q = l_p + N(0, 1), drafts from softmax(q)): the
    first committed token follows p_0 (chi-square, alpha = 1e-3), and the
    acceptance rate at position 0 is sum_v min(p_v, q_v)."""
    rng = np.random.default_rng(7)
    G, V, T = 4, 32, 1.0
    p1 = (rng.standard_normal((G + 1, V)) * 2).astype(np.float32)
    q1 = (p1[:G] + rng.standard_normal((G, V))).astype(np.float32)
    qm = [_softmax(q1[j], T) for j in range(G)]
    counts = np.zeros(V)
    acc0 = 0
    n_total, chunk = 1_000_000, 200_000
    for c0 in range(0, n_total, chunk):
        D = np.stack([rng.choice(V, size=chunk, p=qm[j]) for j in range(G)], 1).astype(np.int32)
        out = oracle_lib.verify(np.broadcast_to(p1, (chunk, 1, G + 1, V)),
                                np.broadcast_to(q1, (chunk, 1, G, V)), D[:, None], T,
                                seed=2024, b0=c0, nthreads=oracle_lib.max_threads())
        L = out["accept_len"]
        first = np.where(L > 0, D[:, 0], out["next_token"])
        counts += np.bincount(first, minlength=V)
        acc0 += int((L > 0).sum())
    p0 = _softmax(p1[0], T)
    expected = p0 * n_total
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp_ = np.append(expected[keep], expected[~keep].sum())
    if exp_[-1] == 0:
        obs, exp_ = obs[:-1], exp_[:-1]
    assert stats.chisquare(obs, exp_).pvalue > 1e-3
    alpha0 = np.minimum(p0, qm[0]).sum()
    assert abs(acc0 / n_total - alpha0) < 5 * np.sqrt(alpha0 * (1 - alpha0) / n_total)


def test_selection_band(oracle_lib):
    """A score that rounding could lift onto the best (or past it) marks the
    selection as boundary; a clear winner or an exact tie of exact ratios does not."""
    V, G = 4, 2
    p = np.zeros((1, 3, G + 1, V), np.float32)
    q = np.zeros((1, 3, G, V), np.float32)
    d = np.zeros((1, 3, G), np.int32)
    # drafts 1 and 2: exact ratio 1 everywhere (q == p); draft 0: ratio 1 - 1e-8
    q[0, 0, 0, 0] = np.float32(1e-8 * 4 / 3)
    out = oracle_lib.verify(p, q, d, 1.0, seed=0)
    assert out["sel"][0] == 1 and out["band"][0] & oracle_lib.BAND_SELECT
    q[0, 0, 0, 0] = 0.5                       # a clear gap: no band
    out = oracle_lib.verify(p, q, d, 1.0, seed=0)
    assert out["sel"][0] == 1 and not out["band"][0] & oracle_lib.BAND_SELECT


def test_data_errors_flagged(oracle_lib):
    rng = np.random.default_rng(8)
    B, K, G, V = 4, 2, 3, 16
    P = rng.standard_normal((B, K, G + 1, V)).astype(np.float32)
    Q = rng.standard_normal((B, K, G, V)).astype(np.float32)
    D = rng.integers(0, V, (B, K, G)).astype(np.int32)
    D[1, 1, 2] = V                      # bad draft id
    P[2, 0, 1, 3] = np.nan              # non-finite row
    T = np.array([1.0, 1.0, 1.0, -1.0])  # bad temperature for b = 3
    out = oracle_lib.verify(P, Q, D, T, seed=0)
    assert list(out["err"]) == [0, oracle_lib.BAD_DRAFT, oracle_lib.BAD_ROW, oracle_lib.BAD_TEMP]
    assert (out["sel"][1:] == -1).all() and (out["next_token"][1:] == -1).all()
    assert out["sel"][0] >= 0
