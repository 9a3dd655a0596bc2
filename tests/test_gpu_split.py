"""The verification step in two calls (sdv_rowpass, then sdv_verify_from_rows)
equals the single call bit for bit: the full layout, greedy acceptance, and
the decode chain's layout (shared marginals and prefix row, the drafter rows'
statistics from the path search, per-sequence lengths), with the path search
running on a second stream while the row pass streams.  One row pass serves
several draft sets.  Misuse is refused before anything is enqueued."""
import numpy as np
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth
from test_gpu_parity import _small, compare, run_oracle

pytestmark = pytest.mark.gpu

KEYS = ("sel", "accept_len", "next_token", "scores", "lse")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def _np(out):
    torch.cuda.synchronize()
    return {k: t.cpu().numpy() for k, t in out.items()}


def _equal(a, b):
    for k in KEYS:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


@pytest.mark.parametrize("greedy", [False, True])
def test_two_calls_equal_one(greedy):
    w = _small(6, 4, 5, 30000, T=0.9, seed=201)
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype, greedy=greedy)
    q = None if greedy else w.q_logits
    one = _np(v(w.p_logits, q, w.drafts, temperature=0.9, seed=4, scores=True, lse=True))
    v.rows(w.p_logits, q, temperature=0.9)
    two = _np(v.finish(w.p_logits, q, w.drafts, temperature=0.9, seed=4, scores=True, lse=True))
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    _equal(one, two)
    if not greedy:
        compare(two, run_oracle(w, seed=4), tag="split full layout")
    v.close()


def test_one_row_pass_serves_several_draft_sets():
    w = _small(4, 3, 6, 20000, T=1.1, seed=202)
    other = w.drafts.flip(1).contiguous()          # the same rows, drafts of another order
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype)
    ref_a = _np(v(w.p_logits, w.q_logits, w.drafts, temperature=1.1, seed=8, scores=True, lse=True))
    ref_b = _np(v(w.p_logits, w.q_logits, other, temperature=1.1, seed=8, scores=True, lse=True))
    v.rows(w.p_logits, w.q_logits, temperature=1.1)
    got_a = _np(v.finish(w.p_logits, w.q_logits, w.drafts, temperature=1.1, seed=8, scores=True, lse=True))
    got_b = _np(v.finish(w.p_logits, w.q_logits, other, temperature=1.1, seed=8, scores=True, lse=True))
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    _equal(ref_a, got_a)
    _equal(ref_b, got_b)
    v.close()


def test_decode_chain_with_the_path_search_on_another_stream():
    """The decode step's layout: the row pass (verifier rows only) on the
    context's stream while the path search runs on a second stream; the rest
    of the step after both, with the search's statistics and lattice lengths."""
    B, K, G, V = 8, 3, 12, 40000
    w = synth.generate_shared(B, K, G, V, q_sigma=torch.full((B, G), 0.6),
                              temps=torch.tensor([0.6, 1.0] * (B // 2)), seed=203, device="cuda")
    eos = 17
    w.q_logits[:, :, eos] = -30.0
    w.q_logits[1, 5, eos] = 30.0                  # one lattice cut short by EOS
    w.q_logits[4, 0, eos] = 30.0
    s_rows, s_cps = torch.cuda.Stream(), torch.cuda.Stream()
    s_rows.wait_stream(torch.cuda.current_stream())
    s_cps.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    # reference: the search, then the single verification call
    cps_ref = bd.sdv_cps(w.q_logits, 0.8, 15, K, eos_id=eos, temps=w.temps, row_stat=True)
    v = bd.Verifier(B, K, G, V, w.dtype, shared_q=True, shared_prefix_row=True)
    # a sequence with fewer distinct paths than the beam has rows of -1: clamp
    # them to a valid id (past the lattice length they are not read)
    ref = _np(v(w.p_logits, w.q_logits, cps_ref["paths"].clamp(min=0).contiguous(), temps=w.temps,
                seed=6, scores=True, lse=True, draft_len=cps_ref["lat_len"],
                q_stat=cps_ref["row_stat"]))
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    # split: row pass on s_rows, path search on s_cps, then the rest on s_rows
    v.set_stream(s_rows)
    with torch.cuda.stream(s_rows):
        v.rows(w.p_logits, w.q_logits, temps=w.temps, with_q=False)
    cps = bd.sdv_cps(w.q_logits, 0.8, 15, K, eos_id=eos, temps=w.temps, row_stat=True, stream=s_cps)
    with torch.cuda.stream(s_cps):
        drafts = cps["paths"].clamp(min=0).contiguous()
    done = torch.cuda.Event()
    done.record(s_cps)
    s_rows.wait_event(done)
    with torch.cuda.stream(s_rows):
        got = v.finish(w.p_logits, w.q_logits, drafts, temps=w.temps, seed=6, scores=True,
                       lse=True, draft_len=cps["lat_len"], q_stat=cps["row_stat"])
    got = _np(got)
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    assert (cps["lat_len"].cpu().numpy() < G).any()
    _equal(ref, got)
    ws = synth.Workload(name="split decode", B=B, K=K, gamma=G, V=V, dtype=w.dtype,
                        p_logits=w.p_logits, q_logits=w.q_logits,
                        drafts=drafts, temperature=1.0,
                        temps=w.temps, seed=6, shared_q=True)
    compare(got, run_oracle(ws, lens=cps["lat_len"].cpu().numpy()), tag="split decode chain")
    v.close()


def test_misuse_is_refused():
    w = _small(2, 2, 3, 4096, seed=204)
    v = bd.Verifier(2, 2, 3, 4096, w.dtype)
    outs = {k: torch.full((2,), -7, dtype=torch.int32, device="cuda") for k in ("sel", "accept_len", "next_token")}

    def finish(q_stat=None, T=1.0, temps=None, lens=None):
        return bd.sdv_verify_from_rows(v.ctx, w.p_logits, w.q_logits, w.drafts, lens, q_stat, T, temps,
                                       0, outs["sel"], outs["accept_len"], outs["next_token"])

    assert finish() == bd.SDV_ERR_ARG and "no row pass" in bd.sdv_last_error(v.ctx)
    assert bd.sdv_rowpass(v.ctx, w.p_logits, w.q_logits, 1.0, None, 0) == bd.SDV_OK
    assert finish() == bd.SDV_ERR_ARG and "q_row_stat" in bd.sdv_last_error(v.ctx)
    assert bd.sdv_rowpass(v.ctx, w.p_logits, w.q_logits, 1.0, None, 1) == bd.SDV_OK
    assert finish(T=0.7) == bd.SDV_ERR_ARG and "temperatures" in bd.sdv_last_error(v.ctx)
    temps = torch.ones(2, device="cuda")
    assert finish(temps=temps) == bd.SDV_ERR_ARG
    # a verify call with lengths skips rows past them: other lengths are refused after it
    lens = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
    v(w.p_logits, w.q_logits, w.drafts, temperature=1.0, draft_len=lens)
    assert finish(lens=torch.tensor([3, 3], dtype=torch.int32, device="cuda")) == bd.SDV_ERR_ARG
    assert finish(lens=lens) == bd.SDV_OK
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    torch.cuda.synchronize()
    v.close()
