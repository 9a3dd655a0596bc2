"""Failure paths of the CUDA library that are tested without faulting or
hanging a GPU.

* The sampling pass's bounded wait for its row copy: with the test hook
  SDV_HOOK_SAMPLE_NO_COPY the kernel arms its barrier but issues no copy, so
  the wait runs out after a few polls with nothing in flight.  The step must
  return, write -1 to every sequence's outputs, and report SDV_ERR_CUDA with
  the timeout text from sdv_sync; the next ordinary step on the same context
  must be correct again.
* Process-wide kernel limits: a context created later for a small vocabulary
  must not lower the shared-memory limit that an earlier large-vocabulary
  context's sampling pass needs.
"""
import numpy as np
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth
from test_gpu_parity import _small, compare, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def _step(v, w, seed):
    out = v(w.p_logits, w.q_logits, w.drafts, temperature=w.temperature, seed=seed, temps=w.temps)
    st = bd.sdv_sync(v.ctx)
    return st, {k: t.cpu().numpy() for k, t in out.items()}


@pytest.mark.parametrize("V", [3000, 152064])
def test_sample_wait_timeout_is_reported_and_the_context_recovers(V):
    B, K, G = 4, 2, 3
    w = _small(B, K, G, V, T=0.9, seed=V + 17)
    v = bd.Verifier(B, K, G, V, w.dtype)
    ok_status, ref = _step(v, w, 5)
    assert ok_status == bd.SDV_OK
    # the hook: barrier armed, no copy issued, a few polls -> the wait gives up
    assert bd.sdv_set_test_hooks(v.ctx, bd.SDV_HOOK_SAMPLE_NO_COPY) == bd.SDV_OK
    st, got = _step(v, w, 5)
    assert st == bd.SDV_ERR_CUDA, bd.STATUS_NAMES.get(st, st)
    assert "bounded device wait gave up" in bd.sdv_last_error(v.ctx)
    for k in ("sel", "accept_len", "next_token"):
        assert (got[k] == -1).all(), (k, got[k])
    # the status was cleared by sdv_sync; normal steps are correct again
    assert bd.sdv_set_test_hooks(v.ctx, 0) == bd.SDV_OK
    st, again = _step(v, w, 5)
    assert st == bd.SDV_OK, bd.sdv_last_error(v.ctx)
    for k in ("sel", "accept_len", "next_token"):
        assert np.array_equal(again[k], ref[k]), k
    assert bd.sdv_set_test_hooks(v.ctx, 2) == bd.SDV_ERR_ARG      # unknown hook bit
    v.close()


def test_a_small_context_does_not_lower_a_large_contexts_limits():
    """The sampling pass of a V = 152064 context needs about 76 KB of dynamic
    shared memory; creating a V = 2000 context afterwards (about 1 KB) must
    leave the earlier context's steps working and correct."""
    big = synth.workload(2, device="cuda")
    vb = bd.Verifier(big.B, big.K, big.gamma, big.V, big.dtype)
    small = _small(2, 2, 3, 2000, seed=3)
    vs = bd.Verifier(2, 2, 3, 2000, small.dtype)
    st_s, _ = _step(vs, small, 1)
    assert st_s == bd.SDV_OK
    out = vb(big.p_logits, big.q_logits, big.drafts, temperature=big.temperature, seed=big.seed,
             scores=True, lse=True)
    assert bd.sdv_sync(vb.ctx) == bd.SDV_OK, bd.sdv_last_error(vb.ctx)
    gpu = {k: t.cpu().numpy() for k, t in out.items()}
    assert compare(gpu, run_oracle(big), tag="large context after a small one") == 0
    vb.close()
    vs.close()
