"""The device adaptive draft length controller (sdv_adl_step, one thread per
sequence) against the oracle's controller, bit-exact over random traces, and
its device-side error report."""
import numpy as np
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


@pytest.mark.parametrize("B,W,kmin,kmax,up,down", [(1, 1, 1, 64, 2, 1), (300, 4, 2, 48, 3, 2),
                                                   (1000, 64, 1, 100, 4, 1)])
def test_device_controller_matches_oracle(B, W, kmin, kmax, up, down):
    import oracle
    rng = np.random.default_rng(B + W)
    ctl = bd.DraftLengthController(B, 0, window=W, kmin=kmin, kmax=kmax, up=up, down=down)
    k = rng.integers(kmin, kmax + 1, B).astype(np.int32)
    ctl.k.copy_(torch.from_numpy(k))
    st = oracle.adl_state(B, W)
    for t in range(120):
        g = np.where(rng.random(B) < 0.7, k, rng.integers(-1, kmax + 2, B)).astype(np.int32)
        a = np.where(rng.random(B) < 0.5, g, rng.integers(-1, kmax + 2, B)).astype(np.int32)
        k = oracle.adl_step(k, g, a, st, W=W, kmin=kmin, kmax=kmax, up=up, down=down)
        got = ctl.step(torch.from_numpy(g).cuda(), torch.from_numpy(a).cuda()).cpu().numpy()
        assert np.array_equal(got, k), t
    assert int(ctl.status.item()) == 0


def test_device_controller_reports_bad_length():
    ctl = bd.DraftLengthController(3, 5, window=2, kmin=2, kmax=8)
    ctl.k[1] = 11
    ctl.step(torch.tensor([5, 5, 3], device="cuda"), torch.tensor([5, 5, 3], device="cuda"))
    torch.cuda.synchronize()
    assert ctl.k.tolist() == [7, 11, 5]               # grown, untouched, held (EOS at 3)
    assert int(ctl.status.item()) & bd.SDV_STATUS_BAD_LENGTH
    L = bd.load()
    host = torch.zeros(3, dtype=torch.int32)
    st = L.sdv_adl_step(3, 2, 2, 8, 2, 1, None, host.data_ptr(), host.data_ptr(), host.data_ptr(),
                        host.data_ptr(), None)
    assert st == bd.SDV_ERR_ARG
    assert L.sdv_adl_step(0, 2, 2, 8, 2, 1, None, None, None, None, None, None) == bd.SDV_OK


def test_decode_step_chain_search_verify_control():
    """One DiffuSpec-style step per iteration, all enqueued on the stream with
    no host synchronisation in between: path search over the marginals ->
    verification of the paths (shared marginals, shared prefix row) ->
    draft-length update from the lattice length and the accepted length.
    Each iteration's lengths are checked against the oracle's controller."""
    import oracle
    from draft_verification_sdv_gb300 import synth
    B, K, G, V = 6, 3, 8, 4000
    ctl = bd.DraftLengthController(B, 6, window=2, kmin=2, kmax=G, up=2, down=1)
    st = oracle.adl_state(B, 2)
    k_ref = np.full(B, 6, np.int32)
    v = bd.Verifier(B, K, G, V, shared_q=True, shared_prefix_row=True)
    gens, accs, ks = [], [], []
    for it in range(3):
        w = synth.generate_shared(B, K, G, V, q_sigma=torch.full((B, G), 0.6), temperature=1.0,
                                  seed=80 + it, device="cuda")
        w.q_logits[:, :, 17] = -30.0
        w.q_logits[1, 5, 17] = 30.0                  # sequence 1 ends at position 5
        cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=K, eos_id=17)
        # each sequence is verified at its lattice length; past it the drafts
        # are not read
        drafts = torch.where(cps["paths"] < 0, torch.zeros_like(cps["paths"]), cps["paths"])
        out = v(w.p_logits, w.q_logits, drafts, temperature=1.0, seed=it, draft_len=cps["lat_len"])
        ks.append(ctl.step(cps["lat_len"], out["accept_len"]).clone())
        gens.append(cps["lat_len"].clone())
        accs.append(out["accept_len"].clone())
    torch.cuda.synchronize()
    v.sync()
    assert all(int(g[1]) == 6 for g in gens) and all((g[[0, 2, 3, 4, 5]] == G).all() for g in gens)
    for g, a, k in zip(gens, accs, ks):
        assert (a <= g).all()                     # nothing past the EOS is accepted
        k_ref = oracle.adl_step(k_ref, g.cpu().numpy(), a.cpu().numpy(), st, W=2, kmin=2, kmax=G,
                                up=2, down=1)
        assert np.array_equal(k.cpu().numpy(), k_ref)
    v.close()
