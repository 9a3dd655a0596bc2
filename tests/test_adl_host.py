"""The library's adaptive draft length controller (host entry point
sdv_adl_step_host, C code in libsdv) against the oracle's, step by step:
next lengths bit-exact over random traces, windows and limits, and the
argument errors.  Runs without a GPU (pure host code of the library)."""
import numpy as np
import pytest
import torch

import oracle
from draft_verification_sdv_gb300 import binding as bd


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bd.load(build=True)


@pytest.mark.parametrize("W,kmin,kmax,up,down", [(1, 1, 64, 2, 1), (3, 2, 20, 3, 2), (8, 4, 100, 5, 5),
                                                 (64, 1, 30, 1, 0), (5, 7, 7, 2, 1)])
def test_host_controller_matches_oracle(W, kmin, kmax, up, down):
    rng = np.random.default_rng(W * 31 + kmax)
    B, steps = 40, 150
    ctl = bd.DraftLengthController(B, 0, window=W, kmin=kmin, kmax=kmax, up=up, down=down, device="cpu")
    k0 = rng.integers(kmin, kmax + 1, B).astype(np.int32)
    ctl.k.copy_(torch.from_numpy(k0))
    st = oracle.adl_state(B, W)
    k = k0.copy()
    for t in range(steps):
        # mostly valid lengths, sometimes out of range (the rule clamps them);
        # some sequences accept everything for a while, some saturate early
        g = np.where(rng.random(B) < 0.7, k, rng.integers(-2, kmax + 3, B)).astype(np.int32)
        a = np.where(rng.random(B) < 0.5, g, rng.integers(-2, kmax + 3, B)).astype(np.int32)
        k = oracle.adl_step(k, g, a, st, W=W, kmin=kmin, kmax=kmax, up=up, down=down)
        got = ctl.step(torch.from_numpy(g), torch.from_numpy(a)).numpy()
        assert np.array_equal(got, k), (t, np.nonzero(got != k))


def test_host_controller_errors():
    L = bd.load()
    assert L.sdv_adl_state_words(0) == -1 and L.sdv_adl_state_words(65) == -1
    assert L.sdv_adl_state_words(3) > 0
    with pytest.raises(bd.SdvError):
        bd.DraftLengthController(2, 4, window=0, device="cpu")
    ctl = bd.DraftLengthController(2, 4, window=2, kmin=2, kmax=8, device="cpu")
    before = ctl.state.clone()
    ctl.k[1] = 9                                     # outside [kmin, kmax]
    with pytest.raises(bd.SdvError):
        ctl.step(torch.tensor([4, 4]), torch.tensor([4, 4]))
    assert torch.equal(ctl.state, before) and ctl.k.tolist() == [4, 9]
    for kw in (dict(kmin=0), dict(kmin=5, kmax=4), dict(up=-1), dict(down=-1), dict(kmax=1 << 21)):
        args = dict(window=1, kmin=1, kmax=8, up=2, down=1)
        args.update(kw)
        st = L.sdv_adl_step_host(1, args["window"], args["kmin"], args["kmax"], args["up"],
                                 args["down"], None, None, None, None)
        assert st == bd.SDV_ERR_ARG, kw


def test_per_sequence_arrays_must_have_B_entries():
    """The library reads B lengths; a shorter or longer array is refused
    before the call."""
    ctl = bd.DraftLengthController(3, 4, window=2, kmin=2, kmax=8, device="cpu")
    with pytest.raises(ValueError):
        ctl.step(torch.tensor([4, 4]), torch.tensor([4, 4, 4]))
    with pytest.raises(ValueError):
        ctl.step(torch.tensor([4, 4, 4]), torch.tensor([4, 4, 4, 4]))
    assert ctl.k.tolist() == [4, 4, 4]
