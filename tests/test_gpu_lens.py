"""Per-sequence draft lengths in the CUDA path (sdv_verify_len) against the
oracle with the same lengths.  The oracle's lengths are pinned by reduction
to each sequence's truncated problem.  Also covered here: full lengths give
the full-length outputs bit for bit; rows and drafts past a length are never
read (NaN / invalid ids there change nothing); the unread rows' LSE entries
are NaN; a length outside [0, gamma] is a data error; and the path-search
lattice lengths feed verification directly."""
import numpy as np
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth
from test_gpu_parity import compare, full_size_bounds, _small

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def _run(w, lens, seed=3, greedy=False, shared_prefix_row=False):
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype, shared_q=w.shared_q and not greedy,
                    greedy=greedy, shared_prefix_row=shared_prefix_row)
    dl = None if lens is None else torch.as_tensor(lens, dtype=torch.int32, device="cuda")
    out = v(w.p_logits, None if greedy else w.q_logits, w.drafts, temperature=w.temperature,
            seed=seed, temps=w.temps, scores=True, lse=True, draft_len=dl)
    status = bd.sdv_sync(v.ctx)
    res = {k: t.cpu().numpy() for k, t in out.items()}
    res["status"] = status
    v.close()
    return res


def _oracle(w, lens, seed=3, greedy=False):
    import oracle
    p, q, d, t = synth.to_oracle_arrays(w)
    if greedy:
        return oracle.verify_greedy(p, d, t, seed, lens=lens, nthreads=oracle.max_threads())
    return oracle.verify(p, q, d, t, seed, lens=lens, nthreads=oracle.max_threads())


def _nan_pattern_agrees(gpu, orc):
    lg = gpu["lse"]
    lo = orc["lse"][..., :lg.shape[-1]]
    ok = orc["err"] == 0
    assert np.array_equal(np.isnan(lg[ok]), np.isnan(lo[ok]))


@pytest.mark.parametrize("greedy", [False, True])
def test_random_lengths_match_oracle(greedy):
    B, K, G, V = 24, 3, 6, 5000
    w = _small(B, K, G, V, T=0.9, seed=31)
    lens = np.array([b % (G + 1) for b in range(B)], np.int32)
    gpu, orc = _run(w, lens, greedy=greedy), _oracle(w, lens, greedy=greedy)
    assert gpu["status"] == bd.SDV_OK
    assert compare(gpu, orc, tag="lens greedy=%s" % greedy) <= 2
    _nan_pattern_agrees(gpu, orc)
    assert ((gpu["accept_len"] >= 0) & (gpu["accept_len"] <= lens)).all()
    assert (gpu["sel"][lens == 0] == 0).all() and (gpu["scores"][lens == 0] == 0).all()


def test_full_lengths_equal_full_step_bitwise():
    w = _small(6, 4, 5, 9000, T=1.1, seed=32)
    ref = _run(w, None)
    got = _run(w, np.full(6, 5, np.int32))
    for k in ("sel", "accept_len", "next_token", "scores", "lse"):
        assert np.array_equal(got[k], ref[k], equal_nan=True), k


def test_rows_and_drafts_past_the_length_are_not_read():
    B, K, G, V = 8, 3, 6, 4000
    w = _small(B, K, G, V, seed=33)
    lens = np.array([0, 1, 2, 3, 4, 5, 6, 3], np.int32)
    ref = _run(w, lens)
    p, q, d = w.p_logits.clone(), w.q_logits.clone(), w.drafts.clone()
    for b, L in enumerate(lens):
        p[b, :, L + 1:] = float("nan")
        q[b, :, L:] = float("nan")
        d[b, :, L:] = -7
    w2 = synth.Workload(name="poisoned", B=B, K=K, gamma=G, V=V, dtype=w.dtype, p_logits=p,
                        q_logits=q, drafts=d, temperature=w.temperature, temps=w.temps,
                        seed=w.seed)
    got = _run(w2, lens)
    assert got["status"] == bd.SDV_OK
    for k in ("sel", "accept_len", "next_token", "scores", "lse"):
        assert np.array_equal(got[k], ref[k], equal_nan=True), k


def test_length_out_of_range_is_a_data_error():
    w = _small(3, 2, 4, 2000, seed=34)
    got = _run(w, np.array([4, 5, -1], np.int32))
    assert got["status"] == bd.SDV_ERR_DEVICE_DATA
    assert got["sel"][0] >= 0 and (got["sel"][1:] == -1).all() and (got["next_token"][1:] == -1).all()
    # through the C ABI: a host buffer, or none, is rejected before any launch
    v = bd.Verifier(3, 2, 4, 2000)
    outs = [torch.empty(3, dtype=torch.int32, device="cuda") for _ in range(3)]
    host = torch.zeros(3, dtype=torch.int32)
    for dl in (host.data_ptr(), None):
        st = bd.load().sdv_verify_len(v.ctx, w.p_logits.data_ptr(), w.q_logits.data_ptr(),
                                      w.drafts.data_ptr(), dl, 1.0, None, 0,
                                      *[o.data_ptr() for o in outs], None, None)
        assert st == bd.SDV_ERR_ARG
    v.close()


def test_lattice_lengths_feed_verification():
    """Paths cut at EOS are verified at their own length: shared marginals,
    the shared prefix row, draft_len = the lattice length."""
    import oracle
    B, K, G, V, eos = 6, 3, 8, 4000, 17
    w = synth.generate_shared(B, K, G, V, q_sigma=torch.full((B, G), 0.6), temperature=1.0,
                              seed=35, device="cuda")
    w.q_logits[:, :, eos] = -30.0
    w.q_logits[1, 4, eos] = 30.0
    w.q_logits[4, 0, eos] = 30.0
    cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=K, eos_id=eos)
    torch.cuda.synchronize()
    assert cps["lat_len"].tolist() == [G, 5, G, G, 1, G]
    w.drafts = torch.where(cps["paths"] < 0, torch.zeros_like(cps["paths"]), cps["paths"]).contiguous()
    lens = cps["lat_len"].cpu().numpy()
    gpu = _run(w, lens, shared_prefix_row=True)
    orc = _oracle(w, lens)
    assert gpu["status"] == bd.SDV_OK
    assert compare(gpu, orc, tag="lattice lengths") <= 1
    # an accepted EOS ends the sequence: nothing after it is accepted
    assert (gpu["accept_len"] <= lens).all()


def test_large_window_random_lengths_full():
    """sdv_verify_len at the large-window size: every sequence against the
    oracle with the same random lengths."""
    w = synth.workload(5, device="cuda", seed=5)
    rng = np.random.default_rng(36)
    lens = rng.integers(0, w.gamma + 1, w.B).astype(np.int32)
    gpu = _run(w, lens, seed=w.seed)
    assert gpu["status"] == bd.SDV_OK
    orc = _oracle(w, lens, seed=w.seed)
    nb = compare(gpu, orc, tag="large-window lens (all 32)",
                 max_kind=full_size_bounds(32))
    assert nb <= 32 // 4 + 6
    _nan_pattern_agrees(gpu, orc)
    del w
    torch.cuda.empty_cache()
