"""sdv_verify_static, the entry point for callers that cannot allocate device
memory -- a process whose device memory belongs to another allocator (a
serving engine's pool), or a plug-in inside such a process -- gives the same
outputs as the context entry point sdv_verify_ex.  It keeps its scratch in a
static device array instead of a context workspace.

Checked through the C ABI on two calls in a row with different shapes, so the
second call runs on scratch the first one left behind.  Outputs are integers:
the tolerance is exact equality, as for every decision in the parity tests.
Once the first call on the device has done its set-up, further calls change
neither torch's allocated memory nor the device's free memory.  Argument
errors -- a host pointer, a misaligned int32 pointer, a shape beyond the
array -- are refused before anything is enqueued.  This file is collected
last so that a stop-at-first-failure run has already run every other test."""
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


def test_static_entry_point_rejects_host_and_misaligned_pointers():
    w = synth.generate(2, 2, 3, 2000, q_sigma=torch.full((2, 2, 3), 0.8), seed=78, device="cuda")
    outs = [torch.full((2,), -7, dtype=torch.int32, device="cuda") for _ in range(3)]
    lib = bd.load()

    def call(p, q, d, o0, o1, o2, temps=None):
        return lib.sdv_verify_static(2, 2, 3, 2000, bd.SDV_BF16, None, p, q, d, 1.0, temps, 0,
                                     o0, o1, o2)

    ptr = [t.data_ptr() for t in (w.p_logits, w.q_logits, w.drafts, *outs)]
    host_drafts = w.drafts.cpu()
    assert call(ptr[0], ptr[1], host_drafts.data_ptr(), *ptr[3:]) == bd.SDV_ERR_ARG
    host_out = torch.zeros(2, dtype=torch.int32)
    assert call(*ptr[:5], host_out.data_ptr()) == bd.SDV_ERR_ARG
    host_p = w.p_logits.cpu()
    assert call(host_p.data_ptr(), *ptr[1:]) == bd.SDV_ERR_ARG
    raw = torch.zeros(16, dtype=torch.int32, device="cuda")
    assert call(*ptr[:2], raw.data_ptr() + 2, *ptr[3:]) == bd.SDV_ERR_ARG     # drafts off by 2 bytes
    assert call(*ptr[:3], raw.data_ptr() + 2, *ptr[4:]) == bd.SDV_ERR_ARG     # out_sel off by 2 bytes
    host_t = torch.ones(2, dtype=torch.float32)
    assert call(*ptr, temps=host_t.data_ptr()) == bd.SDV_ERR_ARG
    torch.cuda.synchronize()
    # nothing was enqueued: the outputs still hold their fill
    assert all((o == -7).all() for o in outs)
    # and the same call with device pointers works
    assert call(*ptr) == bd.SDV_OK
    torch.cuda.synchronize()
    ref = _context_outputs(w, 0)
    for k, o in zip(("sel", "accept_len", "next_token"), outs):
        assert torch.equal(ref[k], o), k


def test_static_calls_allocate_nothing():
    w = synth.generate(6, 4, 5, 30000, q_sigma=torch.full((6, 4, 5), 0.8), seed=79, device="cuda")
    ref = _static_outputs(w, 3)               # the set-up call (first on this device, or not)
    outs = [torch.full((w.B,), -7, dtype=torch.int32, device="cuda") for _ in range(3)]
    args = (w.B, w.K, w.gamma, w.V, bd.SDV_BF16, None, w.p_logits.data_ptr(),
            w.q_logits.data_ptr(), w.drafts.data_ptr(), w.temperature, None, 3,
            *[o.data_ptr() for o in outs])
    lib = bd.load()
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    reserved_before = torch.cuda.memory_reserved()
    free_before, _ = torch.cuda.mem_get_info()
    got = []
    for _ in range(2):
        assert lib.sdv_verify_static(*args) == bd.SDV_OK
        torch.cuda.synchronize()
        got.append([o.cpu() for o in outs])        # device-to-host copies allocate nothing
    free_after, _ = torch.cuda.mem_get_info()
    for call in got:
        for k, o in zip(("sel", "accept_len", "next_token"), call):
            assert torch.equal(ref[k].cpu(), o), k
    assert torch.cuda.memory_allocated() == torch_before
    assert torch.cuda.memory_reserved() == reserved_before
    assert free_after == free_before, (free_before, free_after)
