"""CUDA-graph capture of the device entry points.

A step captured into a graph and replayed gives exactly what the same call
gives when enqueued directly; a replay recomputes from the current contents of
the captured buffers; several steps in one graph (the row pass of a step then
follows the previous step's sampling pass as a programmatic dependent) match
the same steps run one by one; and the whole decode chain (path search ->
verification at the lattice lengths -> draft-length update) captures and
replays with the controller's state advancing as it does eagerly.
"""
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth

pytestmark = pytest.mark.gpu

KEYS = ("sel", "accept_len", "next_token", "scores", "lse")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def _gen(seed, B=6, K=3, G=5, V=5000, T=0.9):
    return synth.generate(B, K, G, V, dtype=torch.bfloat16, p_sigma=3.0, zipf=True,
                          q_sigma=torch.full((B, K, G), 0.8), temperature=T, seed=seed,
                          device="cuda")


def _eager(w, seed, T):
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype)
    out = v(w.p_logits, w.q_logits, w.drafts, temperature=T, seed=seed, scores=True, lse=True)
    v.sync()
    v.close()
    return out


def test_verify_step_captures_and_replays():
    w = _gen(1)
    T = w.temperature
    s = torch.cuda.Stream()
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype, stream=s)
    p, q, d = w.p_logits.clone(), w.q_logits.clone(), w.drafts.clone()
    torch.cuda.synchronize()
    out = v(p, q, d, temperature=T, seed=5, scores=True, lse=True)     # uncaptured first call
    s.synchronize()
    ref = {k: out[k].clone() for k in KEYS}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        v(p, q, d, temperature=T, seed=5, scores=True, lse=True, out=out)
    for k in KEYS:
        out[k].fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(out[k], ref[k]), k
    # new contents in the same buffers: the replay recomputes from them
    w2 = _gen(2)
    p.copy_(w2.p_logits)
    q.copy_(w2.q_logits)
    d.copy_(w2.drafts)
    g.replay()
    torch.cuda.synchronize()
    ref2 = _eager(w2, 5, T)
    for k in KEYS:
        assert torch.equal(out[k], ref2[k]), k
    assert not all(torch.equal(ref[k], ref2[k]) for k in ("sel", "accept_len", "next_token"))
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    v.close()


def test_several_steps_in_one_graph():
    """Three steps back to back in one graph, each with its own inputs, seed
    and outputs, against the same steps run one by one."""
    ws = [_gen(10 + i) for i in range(3)]
    T = ws[0].temperature
    s = torch.cuda.Stream()
    v = bd.Verifier(ws[0].B, ws[0].K, ws[0].gamma, ws[0].V, torch.bfloat16, stream=s)
    torch.cuda.synchronize()
    outs = [v(w.p_logits, w.q_logits, w.drafts, temperature=T, seed=20 + i, scores=True, lse=True)
            for i, w in enumerate(ws)]
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i, w in enumerate(ws):
            v(w.p_logits, w.q_logits, w.drafts, temperature=T, seed=20 + i, scores=True, lse=True,
              out=outs[i])
    for o in outs:
        for k in KEYS:
            o[k].fill_(-7)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for i, w in enumerate(ws):
        ref = _eager(w, 20 + i, T)
        for k in KEYS:
            assert torch.equal(outs[i][k], ref[k]), (i, k)
    v.close()


def test_decode_chain_captures_and_replays():
    """Path search -> verification of the paths at their lattice lengths ->
    draft-length update, captured once and replayed twice, against the same
    chain enqueued directly twice (the controller's window advances the same
    way)."""
    B, K, G, V, eos = 5, 3, 8, 3000, 17
    w = synth.generate_shared(B, K, G, V, q_sigma=torch.full((B, G), 0.6), temperature=1.0,
                              seed=91, device="cuda")
    w.q_logits[:, :, eos] = -30.0
    w.q_logits[2, 4, eos] = 30.0                     # sequence 2 ends at position 4
    s = torch.cuda.Stream()
    torch.cuda.synchronize()

    def make():
        v = bd.Verifier(B, K, G, V, shared_q=True, shared_prefix_row=True, stream=s)
        ctl = bd.DraftLengthController(B, 6, window=2, kmin=2, kmax=G)
        bufs = {"drafts": torch.zeros((B, K, G), dtype=torch.int32, device="cuda")}
        return v, ctl, bufs

    def chain(v, ctl, bufs, cps_out, out):
        cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=K, eos_id=eos, out=cps_out)
        torch.clamp(cps["paths"], min=0, out=bufs["drafts"])
        res = v(w.p_logits, w.q_logits, bufs["drafts"], temperature=1.0, seed=3,
                draft_len=cps["lat_len"], out=out)
        ctl.step(cps["lat_len"], res["accept_len"])
        return cps, res

    # directly, twice
    ve, ce, be = make()
    with torch.cuda.stream(s):
        cps_e, res_e = chain(ve, ce, be, None, None)
        k_first = ce.k.clone()
        chain(ve, ce, be, cps_e, res_e)
    s.synchronize()
    ref = {"paths": cps_e["paths"].clone(), "lat_len": cps_e["lat_len"].clone(),
           "accept_len": res_e["accept_len"].clone(), "next_token": res_e["next_token"].clone(),
           "k": ce.k.clone(), "state": ce.state.clone()}

    # captured: one uncaptured call of each shape first (outputs reused below)
    vg, cg, bg = make()
    with torch.cuda.stream(s):
        cps_g = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=K, eos_id=eos)
        res_g = vg(w.p_logits, w.q_logits, bg["drafts"].clamp(min=0), temperature=1.0, seed=3,
                   draft_len=cps_g["lat_len"])
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain(vg, cg, bg, cps_g, res_g)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(cg.k, k_first)
    g.replay()
    torch.cuda.synchronize()
    got = {"paths": cps_g["paths"], "lat_len": cps_g["lat_len"], "accept_len": res_g["accept_len"],
           "next_token": res_g["next_token"], "k": cg.k, "state": cg.state}
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    assert int(ref["lat_len"][2]) == 5 and (ref["accept_len"] <= ref["lat_len"]).all()
    vg.sync()
    ve.sync()
    vg.close()
    ve.close()
