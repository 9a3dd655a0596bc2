"""Verification with the drafter rows' softmax statistics supplied by the
caller (sdv_verify_qstat), as the path search's pruning pass writes them
(sdv_cps_ex), against the oracle.

The statistics are checked on their own (the row maximum exactly, the sum
against an fp64 sum, the recorded c bit for bit), then the verification that
takes them: against the oracle on the decode chain's shape (paths at their
lattice lengths, shared marginals, shared prefix row) and on the full q
layout; against the same step with the q rows streamed; at the bench's size
on sampled sequences.  A temperature that differs from the one the statistics
were taken at is a data error; greedy contexts and misaligned statistics are
argument errors.
"""
import numpy as np
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth
from test_gpu_parity import compare, full_size_bounds, _small

pytestmark = pytest.mark.gpu

LOG2E = np.float32(1.4426950408889634)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def _shared(B, K, G, V, seed, temps=None, eos=None, cut=()):
    w = synth.generate_shared(B, K, G, V, q_sigma=torch.full((B, G), 0.6), temperature=1.0,
                              temps=temps, seed=seed, device="cuda")
    if eos is not None:
        w.q_logits[:, :, eos] = -30.0
        for b, j in cut:
            w.q_logits[b, j, eos] = 30.0
    return w


def _verify(w, q_stat=None, lens=None, seed=3, shared_prefix_row=False):
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype, shared_q=w.shared_q,
                    shared_prefix_row=shared_prefix_row)
    dl = None if lens is None else torch.as_tensor(lens, dtype=torch.int32, device="cuda")
    out = v(w.p_logits, w.q_logits, w.drafts, temperature=w.temperature, seed=seed, temps=w.temps,
            scores=True, lse=True, draft_len=dl, q_stat=q_stat)
    status = bd.sdv_sync(v.ctx)
    res = {k: t.cpu().numpy() for k, t in out.items()}
    res["status"] = status
    v.close()
    return res


def _oracle(w, lens=None, seed=3, seqs=None):
    import oracle
    p, q, d, t = synth.to_oracle_arrays(w, seqs)
    if seqs is None:
        return oracle.verify(p, q, d, t, seed, lens=lens, nthreads=oracle.max_threads())
    outs = [oracle.verify(p[i:i + 1], q[i:i + 1], d[i:i + 1], t[i:i + 1], seed, b0=b,
                          lens=None if lens is None else lens[b:b + 1],
                          nthreads=oracle.max_threads()) for i, b in enumerate(seqs)]
    return {k: np.concatenate([o[k] for o in outs]) for k in outs[0]}


def test_row_statistics_of_the_pruning_pass():
    B, G, V = 3, 5, 3000
    w = _shared(B, 2, G, V, seed=61, temps=torch.tensor([0.6, 1.0, 1.7]))
    cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=2, temps=w.temps, row_stat=True)
    torch.cuda.synchronize()
    st = cps["row_stat"].cpu().numpy()
    q = w.q_logits.float().cpu().numpy().astype(np.float64)
    T = w.temps.cpu().numpy()
    for b in range(B):
        c = LOG2E / np.float32(T[b])                      # fp32, as the kernels form it
        for j in range(G):
            m = q[b, j].max()
            s = np.sum(np.exp2((q[b, j] - m) * np.float64(c)))
            assert st[b, j, 0] == m
            assert abs(st[b, j, 1] - s) <= 1e-5 * s, (b, j, st[b, j, 1], s)
            assert st[b, j, 2] == c and st[b, j, 3] == 0.0


def test_decode_chain_with_supplied_statistics_matches_oracle():
    """Path search with statistics -> verification of the paths at their
    lattice lengths without streaming the marginals again."""
    B, K, G, V, eos = 8, 3, 8, 4000, 17
    temps = torch.tensor([0.6, 1.0] * 4)
    w = _shared(B, K, G, V, seed=62, temps=temps, eos=eos, cut=((1, 4), (5, 0)))
    cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=K, eos_id=eos, temps=w.temps, row_stat=True)
    torch.cuda.synchronize()
    w.drafts = torch.where(cps["paths"] < 0, torch.zeros_like(cps["paths"]), cps["paths"]).contiguous()
    lens = cps["lat_len"].cpu().numpy()
    assert lens[1] == 5 and lens[5] == 1
    gpu = _verify(w, q_stat=cps["row_stat"], lens=lens, shared_prefix_row=True)
    orc = _oracle(w, lens)
    assert gpu["status"] == bd.SDV_OK
    assert compare(gpu, orc, tag="qstat decode chain") <= 1
    ref = _verify(w, lens=lens, shared_prefix_row=True)   # the same step, q rows streamed
    inside = orc["band"] == 0
    for k in ("sel", "accept_len", "next_token"):
        assert np.array_equal(gpu[k][inside], ref[k][inside]), k


def test_full_q_layout_with_statistics_from_the_pruning_pass():
    """Statistics of [B, K, gamma, V] drafter rows: the pruning half run over
    the rows viewed as B*K sequences, per-sequence temperatures repeated."""
    B, K, G, V = 5, 3, 6, 5000
    temps = torch.tensor([0.7, 1.0, 1.3, 0.9, 1.1], device="cuda")
    w = _small(B, K, G, V, temps=temps, seed=63)
    stat = bd.sdv_cps(w.q_logits.view(B * K, G, V), tau=0.8, mmax=4, beam=1,
                      temps=temps.repeat_interleave(K).contiguous(), row_stat=True)["row_stat"]
    torch.cuda.synchronize()
    lens = np.array([G, 3, 0, G, 5], np.int32)
    gpu = _verify(w, q_stat=stat, lens=lens)
    orc = _oracle(w, lens)
    assert gpu["status"] == bd.SDV_OK
    assert compare(gpu, orc, tag="qstat full layout") <= 1


def test_statistics_of_another_temperature_are_a_data_error():
    B, K, G, V = 4, 2, 5, 3000
    w = _shared(B, K, G, V, seed=64, temps=torch.tensor([1.0, 1.0, 1.0, 1.0]))
    cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=8, beam=K, temps=w.temps, row_stat=True)
    w.drafts = cps["paths"].clamp(min=0).contiguous()
    w.temps = torch.tensor([1.0, 0.7, 1.0, 1.0], device="cuda")     # sequence 1 differs
    gpu = _verify(w, q_stat=cps["row_stat"])
    assert gpu["status"] == bd.SDV_ERR_DEVICE_DATA
    assert gpu["sel"][1] == -1 and gpu["accept_len"][1] == -1 and gpu["next_token"][1] == -1
    assert (gpu["sel"][[0, 2, 3]] >= 0).all()


def test_non_finite_statistics_are_a_bad_row():
    """A supplied row whose max or sum is not finite, or whose sum is not
    positive, is reported like a streamed row holding NaN: that sequence's
    outputs are -1; the others are those of the same step with the rows
    streamed."""
    B, K, G, V = 4, 2, 5, 3000
    w = _shared(B, K, G, V, seed=67)
    cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=8, beam=K, row_stat=True)
    w.drafts = cps["paths"].clamp(min=0).contiguous()
    stat = cps["row_stat"].clone()
    stat[1, 2, 0] = float("nan")                          # sequence 1: NaN max
    stat[3, 0, 1] = 0.0                                   # sequence 3: zero sum
    gpu = _verify(w, q_stat=stat)
    ref = _verify(w)
    assert gpu["status"] == bd.SDV_ERR_DEVICE_DATA
    for b in (1, 3):
        assert gpu["sel"][b] == -1 and gpu["accept_len"][b] == -1 and gpu["next_token"][b] == -1
    orc = _oracle(w)
    for b in (0, 2):
        if orc["band"][b]:
            continue
        for k in ("sel", "accept_len", "next_token"):
            assert gpu[k][b] == ref[k][b], (b, k)


def test_argument_errors():
    B, K, G, V = 2, 2, 4, 512
    w = _shared(B, K, G, V, seed=65)
    stat = torch.zeros((B * G * 4 + 1,), dtype=torch.float32, device="cuda")
    v = bd.Verifier(B, K, G, V, shared_q=True)
    with pytest.raises(bd.SdvError):                       # not 16-byte aligned
        v(w.p_logits, w.q_logits, w.drafts, q_stat=stat[1:])
    with pytest.raises(ValueError):                        # one entry short
        v(w.p_logits, w.q_logits, w.drafts, q_stat=stat[:B * G * 4 - 4])
    with pytest.raises(ValueError):                        # not float32
        v(w.p_logits, w.q_logits, w.drafts, q_stat=stat[:B * G * 4].double())
    with pytest.raises(ValueError):                        # per-sequence arrays of B entries
        v(w.p_logits, w.q_logits, w.drafts, draft_len=torch.zeros(B + 1, dtype=torch.int32,
                                                                  device="cuda"))
    with pytest.raises(ValueError):
        v(w.p_logits, w.q_logits, w.drafts, temps=torch.ones(B - 1, device="cuda"))
    v.close()
    g = bd.Verifier(B, K, G, V, greedy=True)
    with pytest.raises(bd.SdvError):                       # greedy reads no q rows
        g(w.p_logits, None, w.drafts, q_stat=stat[:B * G * 4])
    g.close()


def test_bench_size_full():
    """The decode step's shape: 32 sequences, 3 paths of 32 tokens over
    152064-token marginals, per-sequence temperatures; every sequence against
    the oracle."""
    w = synth.workload_shared(B=32, K=3, gamma=32, device="cuda", seed=66)
    cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=3, temps=w.temps, row_stat=True)
    w.drafts = cps["paths"].clamp(min=0).contiguous()
    lens = cps["lat_len"].cpu().numpy()
    gpu = _verify(w, q_stat=cps["row_stat"], lens=lens, seed=w.seed, shared_prefix_row=True)
    assert gpu["status"] == bd.SDV_OK
    orc = _oracle(w, lens, seed=w.seed)
    nb = compare(gpu, orc, tag="qstat decode-step shape (all 32)",
                 max_kind=full_size_bounds(32))
    assert nb <= 32 // 4 + 6
    del w, cps
    torch.cuda.empty_cache()
