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
