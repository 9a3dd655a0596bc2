"""Pins of the oracle's greedy acceptance mode.

Greedy acceptance ("SpecDiff-2: Scaling Diffusion Drafter Alignment For Faster
Speculative Decoding", section 5.2 and appendix B.4) verifies a draft without
drafter probabilities: token x is accepted when a uniform falls below the
verifier probability p(x); a rejected token is replaced by a draw from p with
the rejected token zeroed out.

Mathematics that pins it: for ANY fixed draft token x, the committed token is
exactly p-distributed, p(x) [v = x] + (1 - p(x)) p(v) [v != x] / (1 - p(x)) =
p(v).  So the committed prefix is an exact autoregressive sample from p
whatever drafts are offered and whichever one the streak score selects:
exhaustive enumeration must return p exactly for K = 1 and K = 2.
"""
import itertools

import numpy as np
import pytest
from scipy import special


def _softmax(l, T):
    return special.softmax(np.asarray(l, np.float64) / T)


def test_greedy_ratio_closed_forms(oracle_lib):
    assert oracle_lib.accept_ratio_greedy(np.log(0.3)) == pytest.approx(0.3, rel=1e-15)
    assert oracle_lib.accept_ratio_greedy(0.0) == 1.0
    assert oracle_lib.accept_ratio_greedy(-np.inf) == 0.0


def test_greedy_acceptance_probability_closed_form(oracle_lib):
    """P(accept position 0) = E_{x~q}[p(x)] = sum_v q_v p_v, through the
    oracle's explicit-uniform entry (u at the interval midpoints)."""
    rng = np.random.default_rng(20)
    G, V, T = 1, 12, 0.9
    p1 = (rng.standard_normal((G + 1, V)) * 1.5).astype(np.float32)
    qm = _softmax(rng.standard_normal(V) * 1.5, 1.0)
    p0 = _softmax(p1[0], T)
    acc = 0.0
    for x in range(V):
        # accepted iff u < p(x): accepted mass is the interval [0, p(x))
        out_a = oracle_lib.verify_greedy_uniforms(p1[None, None], np.array([[[x]]]), T,
                                                  [[p0[x] / 2]], [[0.5, 0.5]])
        out_r = oracle_lib.verify_greedy_uniforms(p1[None, None], np.array([[[x]]]), T,
                                                  [[(1 + p0[x]) / 2]], [[0.5, 0.5]])
        assert out_a["accept_len"][0] == 1 and out_r["accept_len"][0] == 0
        acc += qm[x] * p0[x]
    assert acc == pytest.approx(float(qm @ p0), rel=1e-12)
    assert oracle_lib.verify_greedy(p1[None, None], np.array([[[3]]]), T, 0)["ratio"][0, 0, 0] == \
        pytest.approx(p0[3], rel=1e-12)


def _greedy_branches(p_rows, draft, T):
    """(L, weight, u, [(w, weight, token)]) over the acceptance branches of one
    draft under greedy acceptance, from the test's own softmax."""
    G = len(draft)
    probs = [_softmax(p_rows[j], T) for j in range(G + 1)]
    a = [probs[j][draft[j]] for j in range(G)]
    out, prefix = [], 1.0
    for L in range(G + 1):
        if L < G:
            wt = prefix * (1.0 - a[L])
            u = [a[i] / 2 for i in range(L)] + [(1 + a[L]) / 2] + [0.5] * (G - L - 1)
            r = probs[L].copy()
            r[draft[L]] = 0.0
            prefix *= a[L]
        else:
            wt = prefix
            u = [a[i] / 2 for i in range(G)]
            r = probs[G]
        if wt <= 0 or r.sum() <= 0:
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


@pytest.mark.parametrize("K", [1, 2])
def test_greedy_lossless_exhaustive_with_selection(oracle_lib, K):
    """Every committed token, given that the step reaches it and the committed
    prefix, follows the verifier's conditional exactly -- with self-selection
    among K drafts (V <= 5, gamma <= 2; verifier rows depend on the prefix,
    drafter marginals on the position only)."""
    rng = np.random.default_rng(21 + K)
    for V, G, T in [(3, 1, 1.0), (4, 2, 0.8), (5, 2, 1.3)]:
        vrow = {}

        def verifier_row(prefix):
            if prefix not in vrow:
                vrow[prefix] = (rng.standard_normal(V) * 1.5).astype(np.float32)
            return vrow[prefix]

        qm = [_softmax(rng.standard_normal(V) * 1.5, 1.0) for _ in range(G)]
        per_draft = list(itertools.product(range(V), repeat=G))
        cases, meta = [], []
        for xs in itertools.product(per_draft, repeat=K):
            px = np.prod([qm[j][x[j]] for x in xs for j in range(G)])
            P = np.stack([np.stack([verifier_row(tuple(x[:j])) for j in range(G + 1)]) for x in xs])
            D = np.array(xs, np.int32)
            sel = oracle_lib.verify_greedy_uniforms(P[None], D[None], T, np.zeros((1, G)),
                                                    np.zeros((1, G + 1)))["sel"][0]
            for L, wt, u, draws in _greedy_branches(P[sel], xs[sel], T):
                for wv, wwt, v in draws:
                    W = [0.5] * (G + 1)
                    W[L] = wv
                    cases.append((px * wt * wwt, P, D, u, W))
                    meta.append((xs[sel], L, v, sel))
        out = oracle_lib.verify_greedy_uniforms(
            np.stack([c[1] for c in cases]), np.stack([c[2] for c in cases]), T,
            np.array([c[3] for c in cases]).reshape(len(cases), G), np.array([c[4] for c in cases]))
        law = {}
        for (x, L, v, sel), c, os_, ol, ot in zip(meta, cases, out["sel"], out["accept_len"],
                                                   out["next_token"]):
            assert (os_, ol, ot) == (sel, L, v)
            y = tuple(x[:L]) + (v,)
            law[y] = law.get(y, 0.0) + c[0]
        assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
        for n in range(G + 1):
            for pre in {y[:n] for y in law if len(y) > n}:
                mass = np.zeros(V)
                for y, m in law.items():
                    if len(y) > n and y[:n] == pre:
                        mass[y[n]] += m
                np.testing.assert_allclose(mass / mass.sum(), _softmax(verifier_row(pre), T),
                                           rtol=0, atol=1e-12)


def test_greedy_expected_streak_equals_mean_accepted_length(oracle_lib):
    rng = np.random.default_rng(23)
    G, V, N = 5, 16, 100_000
    p1 = (rng.standard_normal((G + 1, V)) * 1.2).astype(np.float32)
    p1[:, 0] += 3.0                              # a likely token at every position
    x = np.array([0, 0, 1, 0, 0], np.int32)      # mostly the likely token, one unlikely
    out = oracle_lib.verify_greedy(np.broadcast_to(p1, (N, 1, G + 1, V)),
                                   np.broadcast_to(x, (N, 1, G)), 1.0, seed=13,
                                   nthreads=oracle_lib.max_threads())
    S = out["scores"][0, 0]
    L = out["accept_len"].astype(np.float64)
    assert 0.2 < S < G - 0.2
    assert abs(L.mean() - S) < 5 * L.std() / np.sqrt(N)
    # the rejected token is never the replacement
    rej = out["accept_len"] < G
    assert (out["next_token"][rej] != x[out["accept_len"][rej]]).all()
