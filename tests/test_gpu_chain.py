"""The decode chain as the bench runs it, with nothing between the kernels:
path search (its paths fed straight to the verification, which also takes the
search's row statistics) -> verification -> draft-length update, four steps
back to back on one stream.  Every launch but the beam is a programmatic
dependent of the one before and the beam releases its dependents at its
start, so each grid may be resident before the one it depends on ends.  The
outputs must equal, bit for bit, the same chain run with the host waiting
for the device between the search, the verification and the update, and the
verification must equal the oracle on the search's paths."""
import numpy as np
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth
from test_gpu_parity import compare, run_oracle

pytestmark = pytest.mark.gpu

KEYS = ("sel", "accept_len", "next_token", "scores", "lse")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def _chain(ws, temps, sync):
    B, K, G, V = ws[0].B, ws[0].K, ws[0].gamma, ws[0].V
    v = bd.Verifier(B, K, G, V, ws[0].dtype, shared_q=True, shared_prefix_row=True)
    ctl = bd.DraftLengthController(B, G, window=2, kmin=2, kmax=G, up=2, down=1)
    steps = []
    for i, w in enumerate(ws):
        cps = bd.sdv_cps(w.q_logits, 0.8, 15, K, temps=temps, row_stat=True)
        if sync:
            torch.cuda.synchronize()
        out = v(w.p_logits, w.q_logits, cps["paths"], seed=i, temps=temps, scores=True, lse=True,
                draft_len=cps["lat_len"], q_stat=cps["row_stat"])
        if sync:
            torch.cuda.synchronize()
        k = ctl.step(cps["lat_len"], out["accept_len"]).clone()
        if sync:
            torch.cuda.synchronize()
        steps.append(({key: t.clone() for key, t in out.items()},
                      {key: t.clone() for key, t in cps.items()}, k))
    torch.cuda.synchronize()
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    v.close()
    return steps


def test_chained_decode_steps_equal_the_synchronised_chain_and_the_oracle():
    B, K, G, V = 12, 3, 10, 6000
    temps = torch.tensor([0.6, 1.0, 1.3] * (B // 3), device="cuda")
    ws = [synth.generate_shared(B, K, G, V, q_sigma=torch.full((B, G), 0.8), temps=temps.cpu(),
                                seed=400 + i, device="cuda") for i in range(4)]
    fast = _chain(ws, temps, sync=False)
    slow = _chain(ws, temps, sync=True)
    for (of, cf, kf), (os_, cs, ks) in zip(fast, slow):
        assert (cf["npaths"] == K).all()          # every draft row is a real path
        for key in cf:
            assert torch.equal(cf[key], cs[key]), key
        for key in KEYS:
            assert np.array_equal(of[key].cpu().numpy(), os_[key].cpu().numpy(), equal_nan=True), key
        assert torch.equal(kf, ks)
    # the last step's verification against the oracle on its paths
    w, (out, cps, _) = ws[-1], fast[-1]
    wd = synth.Workload(name="chained decode", B=B, K=K, gamma=G, V=V, dtype=w.dtype,
                        p_logits=w.p_logits, q_logits=w.q_logits, drafts=cps["paths"],
                        temperature=1.0, temps=temps.cpu(), seed=len(ws) - 1, shared_q=True)
    gpu = {key: t.cpu().numpy() for key, t in out.items()}
    compare(gpu, run_oracle(wd, lens=cps["lat_len"].cpu().numpy()), tag="chained decode step")
