"""Pins of the oracle's causal-consistency path search ("DiffuSpec: Unlocking
Diffusion Language Models for Speculative Decoding", section 4.2: prune each
position's candidates by cumulative probability mass, stop at the first EOS,
beam-search left to right on the pruned lattice; section 5.3: beam 3, at most
15 candidates, mass 0.8).

The pruning is pinned by the invariants that characterise the kept set (not
by re-sorting): its mass reaches tau unless the cap binds, dropping its last
member falls below tau, and every kept token is at least as likely as every
dropped one.  The beam is pinned by brute force: with a score that adds
per-position log-probabilities, the beam must return the exact best paths of
the whole lattice.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest
from scipy import special


def _probs(row, T):
    return special.softmax(np.asarray(row, np.float64) / T)


@pytest.mark.parametrize("V,T,tau,mmax", [(12, 1.0, 0.8, 15), (40, 0.7, 0.5, 5), (9, 2.0, 0.99, 9),
                                          (30, 1.0, 1.0, 4), (20, 0.5, 0.0, 3)])
def test_prune_invariants(oracle_lib, V, T, tau, mmax):
    rng = np.random.default_rng(V + mmax)
    for trial in range(20):
        row = (rng.standard_normal(V) * 2).astype(np.float32)
        if trial % 4 == 0:
            row[rng.integers(0, V, 3)] = row[0]            # exact ties
        ids, lp, before, after = oracle_lib.cps_prune_row(row, T, tau, mmax)
        p = _probs(row, T)
        n = len(ids)
        assert 1 <= n <= mmax
        np.testing.assert_allclose(np.exp(lp), p[ids], rtol=1e-12)
        assert after == pytest.approx(p[ids].sum(), rel=1e-12)
        assert after >= tau or n == mmax                  # reaches tau unless capped
        assert before < tau or n == 1                     # minimal: the last token was needed
        dropped = np.setdiff1d(np.arange(V), ids)
        if len(dropped):
            assert p[ids].min() >= p[dropped].max()       # kept dominate dropped
        # order: probability descending, ties by lower id
        for a, b in zip(ids[:-1], ids[1:]):
            assert p[a] > p[b] or (p[a] == p[b] and a < b)


def _lattice_best(q_b, cand_ids, ncand, L, W):
    """All paths of the lattice, best first, in exact arithmetic: a path's
    score is sum_j (l_j(x_j) / T - lse_j), so with T and the lse_j common to
    every path the order is that of the exact sum of the raw logits
    (fractions); equal sums go to the lexicographically first candidate
    ranks."""
    paths = []
    for ranks in itertools.product(*[range(ncand[j]) for j in range(L)]):
        key = sum(Fraction(float(q_b[j, cand_ids[j, r]])) for j, r in enumerate(ranks))
        paths.append((-key, ranks))
    paths.sort()
    return paths[:W]


@pytest.mark.parametrize("W", [1, 3, 7])
@pytest.mark.parametrize("grid", [False, True])
def test_beam_is_exact_top_paths(oracle_lib, W, grid):
    """With logits on a coarse grid (as bf16 logits are) many paths tie
    exactly; the tie rule must then decide, not rounding."""
    rng = np.random.default_rng(30 + W + 10 * grid)
    B, G, V, T = 6, 4, 10, 0.7
    q = (rng.standard_normal((B, G, V)) * 1.5).astype(np.float32)
    if grid:
        q = np.round(q * 4) / 4
    q[0, 1, :3] = 2.0                                        # tied candidates
    out = oracle_lib.cps(q, T, 0.9, 4, W)
    for b in range(B):
        L = out["lat_len"][b]
        assert L == G
        best = _lattice_best(q[b], out["cand_ids"][b], out["ncand"][b], L, W)
        assert out["npaths"][b] == len(best)
        for w, (negkey, ranks) in enumerate(best):
            ids = [out["cand_ids"][b, j, r] for j, r in enumerate(ranks)]
            assert list(out["paths"][b, w, :L]) == ids
            # the reported score is the path's log-probability
            lp = sum(np.log(_probs(q[b, j], T)[i]) for j, i in enumerate(ids))
            assert out["path_logp"][b, w] == pytest.approx(lp, rel=1e-12, abs=1e-12)


def test_eos_cuts_the_lattice(oracle_lib):
    B, G, V, eos = 2, 5, 16, 7
    rng = np.random.default_rng(40)
    q = rng.standard_normal((B, G, V)).astype(np.float32)
    q[0, :2, eos] = -9.0
    q[0, 2, eos] = 9.0                                       # EOS first most likely at position 2
    q[1, :, eos] = -9.0                                      # never EOS
    out = oracle_lib.cps(q, 1.0, 0.8, 6, 3, eos_id=eos)
    assert list(out["lat_len"]) == [3, G]
    assert out["ncand"][0, 2] == 1 and (out["ncand"][0, 3:] == 0).all()
    for w in range(out["npaths"][0]):
        assert out["paths"][0, w, 2] == eos and (out["paths"][0, w, 3:] == -1).all()
    assert (out["paths"][1, :out["npaths"][1]] >= 0).all()


def test_single_candidate_lattice_is_argmax(oracle_lib):
    """tau = 0: one candidate per position, the argmax; one path."""
    rng = np.random.default_rng(41)
    q = rng.standard_normal((3, 6, 50)).astype(np.float32)
    out = oracle_lib.cps(q, 1.0, 0.0, 8, 4)
    assert (out["ncand"] == 1).all() and (out["npaths"] == 1).all()
    assert (out["paths"][:, 0] == q.argmax(-1)).all()


def test_zero_probability_tokens_and_bad_rows(oracle_lib):
    """A token of probability zero (logit -inf) adds no mass and is never a
    candidate; a row with a NaN or +inf logit, or with no finite logit, has no
    probability distribution and offers no candidates, so no path exists."""
    row = np.full(20, -np.inf, np.float32)
    row[[4, 9, 13]] = [1.0, 3.0, 2.0]
    ids, lp, before, after = oracle_lib.cps_prune_row(row, 1.0, 1.0, 15)
    assert list(ids) == [9, 13, 4]                     # all finite tokens, nothing else
    assert after == pytest.approx(1.0, rel=1e-14)
    np.testing.assert_allclose(np.exp(lp), _probs(row[[9, 13, 4]], 1.0), rtol=1e-12)
    for bad in (np.nan, np.inf):
        r2 = row.copy()
        r2[0] = bad
        assert len(oracle_lib.cps_prune_row(r2, 1.0, 0.8, 15)[0]) == 0
    assert len(oracle_lib.cps_prune_row(np.full(8, -np.inf, np.float32), 1.0, 0.8, 15)[0]) == 0
    q = np.random.default_rng(42).standard_normal((2, 3, 16)).astype(np.float32)
    q[1, 1, 5] = np.nan
    out = oracle_lib.cps(q, 1.0, 0.8, 6, 3)
    assert out["ncand"][1, 1] == 0 and out["npaths"][1] == 0
    assert (out["paths"][1] == -1).all() and np.isneginf(out["path_logp"][1]).all()
    assert out["npaths"][0] >= 1
