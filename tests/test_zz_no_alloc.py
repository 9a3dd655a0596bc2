"""sdv_verify_static, the entry point for callers that cannot allocate device
memory (it keeps its scratch in a static device array instead of a context
workspace), gives the same outputs as the context entry point sdv_verify_ex.

Checked through the C ABI on two calls in a row with different shapes, so the
second call runs on scratch the first one left behind.  Outputs are integers:
the tolerance is exact equality, as for every decision in the parity tests.
This file is collected last so that a stop-at-first-failure run has already
run every other test."""
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def _context_outputs(w, seed):
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype)
    out = v(w.p_logits, w.q_logits, w.drafts, temperature=w.temperature, seed=seed, temps=w.temps)
    v.sync()
    res = {k: t.clone() for k, t in out.items()}
    v.close()
    return res


def _static_outputs(w, seed):
    out = {k: torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
           for k in ("sel", "accept_len", "next_token")}
    st = bd.sdv_verify_static(w.B, w.K, w.gamma, w.V, w.dtype, None, w.p_logits, w.q_logits,
                              w.drafts, w.temperature, w.temps, seed, out["sel"],
                              out["accept_len"], out["next_token"])
    assert st == bd.SDV_OK, bd.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    return out


def test_static_entry_point_matches_context_entry_point():
    # call 1: the self-selection workload (8 x 4 drafts of 16, Qwen vocabulary)
    w1 = synth.workload(3, device="cuda")
    # call 2: a smaller shape with per-sequence temperatures, on the scratch
    # the first call left behind
    w2 = synth.generate(5, 3, 6, 20000, q_sigma=torch.full((5, 3, 6), 0.9),
                        temps=torch.tensor([0.6, 1.0, 1.3, 0.8, 1.0]), seed=77, device="cuda")
    for w, seed in ((w1, 11), (w2, 12)):
        ref = _context_outputs(w, seed)
        got = _static_outputs(w, seed)
        for k in ("sel", "accept_len", "next_token"):
            assert torch.equal(ref[k], got[k]), k
    # and once more on the first shape after the second
    assert all(torch.equal(_context_outputs(w1, 11)[k], _static_outputs(w1, 11)[k])
               for k in ("sel", "accept_len", "next_token"))


def test_static_entry_point_rejects_oversized_shapes():
    dummy = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    outs = [torch.zeros(4, dtype=torch.int32, device="cuda") for _ in range(3)]
    d = torch.zeros(4, dtype=torch.int32, device="cuda")
    # 2.1 million rows need more than 8 MiB of partials even at one chunk per row
    st = bd.sdv_verify_static(1000, 64, 16, 64, torch.bfloat16, None, dummy, dummy, d, 1.0, None,
                              0, *outs)
    assert st == bd.SDV_ERR_SCRATCH
    # a million sequences' tasks alone exceed the array
    st = bd.sdv_verify_static(1 << 20, 1, 1, 64, torch.bfloat16, None, dummy, dummy, d, 1.0, None,
                              0, *outs)
    assert st == bd.SDV_ERR_SCRATCH
    st = bd.sdv_verify_static(4, 1, 1, 64, torch.bfloat16, None, dummy, dummy, d, 0.0, None, 0, *outs)
    assert st == bd.SDV_ERR_ARG
