"""Pins of the oracle's adaptive draft length controller ("DiffuSpec:
Unlocking Diffusion Language Models for Speculative Decoding", section 4.3
and appendix C: the draft length grows while accepted length keeps pace with
the EOS-aware generated length, and stops growing as the generated length
saturates).

The page gives the direction of the rule, not a formula; the reading pinned
here: over the last W steps, acceptance keeps pace when the accepted lengths
sum to the generated ones, generation fills the drafts when the generated
lengths sum to the drafted ones; keep pace and fill -> grow by `up`; keep pace
but saturate -> hold; fall behind -> shrink by `down`; clamp to [kmin, kmax].
The traces below are worked by hand from that statement."""
import numpy as np
import pytest


def _run(oracle_lib, k0, steps, **kw):
    W = kw.get("W", 1)
    st = oracle_lib.adl_state(1, W)
    k, out = np.array([k0]), []
    for g, a in steps:
        k = oracle_lib.adl_step(k, [g], [a], st, **kw)
        out.append(int(k[0]))
    return out, st


def test_single_step_window_trace(oracle_lib):
    # full acceptance grows 4 -> 6 -> 8 -> 10 (cap 10), a rejection shrinks by
    # one, an EOS-short draft fully accepted holds, a rejection shrinks again
    steps = [(4, 4), (6, 6), (8, 8), (10, 10), (10, 3), (5, 5), (9, 2)]
    got, _ = _run(oracle_lib, 4, steps, W=1, kmin=1, kmax=10, up=2, down=1)
    assert got == [6, 8, 10, 10, 9, 9, 8]


def test_window_of_three_trace(oracle_lib):
    # (k, g, a) per step; sums over the last three decide
    #  1: (8,8,8)                          k 8  g 8  a 8  -> grow  11
    #  2: (11,11,5)                        k19  g19  a13  -> shrink 9
    #  3: (9,9,9)                          k28  g28  a22  -> shrink 7
    #  4: (7,7,7), (8,8,8) leaves          k27  g27  a21  -> shrink 5
    #  5: (5,5,5)                          k21  g21  a21  -> grow   8
    #  6: (8,4,4)   EOS at 4               k20  g16  a16  -> hold   8
    #  7: (8,12->8, 9->8) clamped          k21  g17  a17  -> hold   8
    #  8: (8,8,-1->0)                      k24  g20  a12  -> shrink 6
    steps = [(8, 8), (11, 5), (9, 9), (7, 7), (5, 5), (4, 4), (12, 9), (8, -1)]
    got, st = _run(oracle_lib, 8, steps, W=3, kmin=2, kmax=20, up=3, down=2)
    assert got == [11, 9, 7, 5, 8, 8, 8, 6]
    assert 3 <= st[0, 0] < 6                     # the step counter stays bounded


def test_floor_and_cap(oracle_lib):
    got, _ = _run(oracle_lib, 3, [(3, 0), (2, 0), (2, 1)], W=1, kmin=2, kmax=9, up=5, down=2)
    assert got == [2, 2, 2]
    got, _ = _run(oracle_lib, 7, [(7, 7), (9, 9)], W=1, kmin=2, kmax=9, up=5, down=2)
    assert got == [9, 9]


def test_invalid_parameters(oracle_lib):
    st = oracle_lib.adl_state(1, 2)
    for kw in (dict(W=0), dict(kmin=0), dict(kmin=5, kmax=4), dict(up=-1), dict(down=-1)):
        with pytest.raises(ValueError):
            oracle_lib.adl_step([4], [4], [4], oracle_lib.adl_state(1, max(kw.get("W", 2), 1)),
                                **{"W": 2, **kw})
    with pytest.raises(ValueError):                # a k outside [kmin, kmax]
        oracle_lib.adl_step([70], [4], [4], st, W=2, kmin=1, kmax=64)


def test_batch_equals_sequences_one_by_one_and_step_invariants(oracle_lib):
    rng = np.random.default_rng(5)
    B, W, kmin, kmax, up, down = 12, 4, 2, 40, 3, 2
    stB = oracle_lib.adl_state(B, W)
    st1 = [oracle_lib.adl_state(1, W) for _ in range(B)]
    k = rng.integers(kmin, kmax + 1, B).astype(np.int32)
    k1 = [np.array([x]) for x in k]
    for _ in range(60):
        g = np.minimum(k, rng.integers(0, kmax + 5, B)).astype(np.int32)
        a = np.minimum(g, rng.integers(0, kmax + 5, B)).astype(np.int32)
        nk = oracle_lib.adl_step(k, g, a, stB, W=W, kmin=kmin, kmax=kmax, up=up, down=down)
        for b in range(B):
            k1[b] = oracle_lib.adl_step(k1[b], [g[b]], [a[b]], st1[b], W=W, kmin=kmin,
                                        kmax=kmax, up=up, down=down)
            assert k1[b][0] == nk[b]
            # one move of the rule, then the clamp
            assert nk[b] in {min(kmax, k[b] + up), k[b], max(kmin, k[b] - down)}
        assert ((nk >= kmin) & (nk <= kmax)).all()
        k = nk
    for b in range(B):
        assert np.array_equal(st1[b][0], stB[b])


def test_more_acceptance_never_shortens_the_next_draft(oracle_lib):
    rng = np.random.default_rng(6)
    for _ in range(200):
        W = int(rng.integers(1, 5))
        hist = [(int(kk), int(gg), int(aa)) for kk, gg, aa in rng.integers(1, 20, (W - 1, 3))]
        k0 = int(rng.integers(1, 30))
        g = int(rng.integers(0, k0 + 1))
        res = []
        for a in range(g + 1):
            st = oracle_lib.adl_state(1, W)
            for kk, gg, aa in hist:
                kk = min(kk, 30)
                oracle_lib.adl_step([kk], [gg], [aa], st, W=W, kmin=1, kmax=30)
            res.append(int(oracle_lib.adl_step([k0], [g], [a], st, W=W, kmin=1, kmax=30)[0]))
        assert res == sorted(res)


def test_inputs_are_clamped(oracle_lib):
    # a generated length above the draft counts as the draft: (8, 12, 8) is a
    # fully accepted full draft -> grow
    got, _ = _run(oracle_lib, 8, [(12, 8)], W=1, kmin=1, kmax=20, up=2, down=1)
    assert got == [10]
    # an accepted length above the generated one counts as the generated one:
    # window (8,8,4), (8,8,12->8): a 12 < g 16 -> shrink
    got, _ = _run(oracle_lib, 8, [(8, 4), (8, 12)], W=2, kmin=1, kmax=20, up=2, down=1)
    assert got == [7, 6]
