"""Pins of the oracle's per-sequence draft lengths.

A batch whose sequences carry drafts of different lengths (an adaptive draft
length, or paths cut at EOS; "DiffuSpec: Unlocking Diffusion Language Models
for Speculative Decoding", sections 4.2-4.3) must verify each sequence exactly
as the full-length algorithm verifies its drafts truncated to that length:
the same rows, the same uniforms (keyed by position and sequence), the bonus
token from the verifier row right after the last draft token.  The
full-length algorithm is pinned elsewhere; these tests reduce to it."""
import numpy as np
import pytest


def _case(rng, B, K, G, V):
    p = (rng.standard_normal((B, K, G + 1, V)) * 1.5).astype(np.float32)
    q = (p[:, :, :G] + rng.standard_normal((B, K, G, V)) * 0.8).astype(np.float32)
    d = rng.integers(0, V, (B, K, G)).astype(np.int32)
    t = rng.uniform(0.6, 1.4, B)
    return p, q, d, t


KEYS = ("sel", "accept_len", "next_token", "scores", "err")


@pytest.mark.parametrize("greedy", [False, True])
def test_full_length_equals_no_lengths(oracle_lib, greedy):
    rng = np.random.default_rng(70 + greedy)
    p, q, d, t = _case(rng, 6, 3, 5, 40)
    if greedy:
        a = oracle_lib.verify_greedy(p, d, t, 9)
        b = oracle_lib.verify_greedy(p, d, t, 9, lens=np.full(6, 5))
    else:
        a = oracle_lib.verify(p, q, d, t, 9)
        b = oracle_lib.verify(p, q, d, t, 9, lens=np.full(6, 5))
    for k in KEYS + ("lse",):
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("greedy", [False, True])
def test_each_sequence_equals_its_truncated_problem(oracle_lib, greedy):
    """Sequence b with length L_b gives what the full-length algorithm gives
    on its drafts cut to L_b (same b in the uniform keying); every length
    0..gamma occurs."""
    rng = np.random.default_rng(72 + greedy)
    B, K, G, V = 14, 3, 6, 30
    p, q, d, t = _case(rng, B, K, G, V)
    lens = np.array([b % (G + 1) for b in range(B)], np.int32)
    if greedy:
        out = oracle_lib.verify_greedy(p, d, t, 11, lens=lens)
    else:
        out = oracle_lib.verify(p, q, d, t, 11, lens=lens)
    for b in range(B):
        L = int(lens[b])
        pb = np.ascontiguousarray(p[b:b + 1, :, :L + 1])
        qb = np.ascontiguousarray(q[b:b + 1, :, :L])
        db = np.ascontiguousarray(d[b:b + 1, :, :L])
        if greedy:
            ref = oracle_lib.verify_greedy(pb, db, t[b:b + 1], 11, b0=b)
        else:
            ref = oracle_lib.verify(pb, qb, db, t[b:b + 1], 11, b0=b)
        for k in KEYS:
            assert out[k][b] == ref[k][0] if np.ndim(out[k][b]) == 0 else \
                np.array_equal(out[k][b], ref[k][0]), (b, k)
        assert 0 <= out["accept_len"][b] <= L
        # the rows that are read agree; the others are reported as NaN
        G1 = G + 1
        np.testing.assert_array_equal(out["lse"][b][:, :L + 1], ref["lse"][0][:, :L + 1])
        assert np.isnan(out["lse"][b][:, L + 1:G1]).all()
        if not greedy:
            np.testing.assert_array_equal(out["lse"][b][:, G1:G1 + L], ref["lse"][0][:, L + 1:])
            assert np.isnan(out["lse"][b][:, G1 + L:]).all()


def test_rows_past_the_length_are_not_read(oracle_lib):
    rng = np.random.default_rng(74)
    B, K, G, V = 5, 2, 6, 25
    p, q, d, t = _case(rng, B, K, G, V)
    lens = np.array([0, 2, 3, 5, 6], np.int32)
    ref = oracle_lib.verify(p, q, d, t, 5, lens=lens)
    p2, q2, d2 = p.copy(), q.copy(), d.copy()
    for b, L in enumerate(lens):
        p2[b, :, L + 1:] = np.nan
        q2[b, :, L:] = np.nan
        d2[b, :, L:] = -7                     # invalid ids past the length are never looked at
    got = oracle_lib.verify(p2, q2, d2, t, 5, lens=lens)
    for k in KEYS:
        np.testing.assert_array_equal(got[k], ref[k])


def test_zero_length_draws_from_the_prefix_row(oracle_lib):
    """No drafts: nothing to select or accept; the token is a draw from the
    verifier row at position 0 with the uniform w_0 (the bonus rule at L = 0)."""
    rng = np.random.default_rng(75)
    B, K, G, V = 4, 3, 4, 12
    p, q, d, t = _case(rng, B, K, G, V)
    out = oracle_lib.verify(p, q, d, t, 21, lens=np.zeros(B, np.int32))
    assert (out["sel"] == 0).all() and (out["accept_len"] == 0).all()
    assert (out["scores"] == 0).all()
    for b in range(B):
        probs = np.exp(p[b, 0, 0] / t[b] - np.logaddexp.reduce(p[b, 0, 0] / t[b]))
        _, w = oracle_lib.uniforms(21, b, 0)
        c = np.cumsum(probs)
        assert out["next_token"][b] == int(np.argmax(c > w * c[-1]))


def test_length_out_of_range_is_an_error(oracle_lib):
    rng = np.random.default_rng(76)
    p, q, d, t = _case(rng, 3, 2, 4, 10)
    out = oracle_lib.verify(p, q, d, t, 1, lens=np.array([4, 5, -1], np.int32))
    assert out["err"][0] == 0 and out["err"][1] != 0 and out["err"][2] != 0
    assert (out["sel"][1:] == -1).all() and (out["next_token"][1:] == -1).all()
