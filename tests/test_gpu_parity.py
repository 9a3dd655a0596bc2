"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Bar (decisions are integers): selected draft, accepted length and emitted
token bit-exact, except trials the oracle flags inside the 1e-5 boundary band
(a uniform within 1e-5 relative of an acceptance ratio or CDF boundary; a
selection that a 1e-5 relative move of any p/q could reorder; residual mass
below 1e-3), which are counted and reported.
Row LSE and expected-streak scores within 1e-4 relative (LSE against
max(1, |LSE|)).
"""
import numpy as np
import pytest
import torch

import band_report
from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth

pytestmark = pytest.mark.gpu

LSE_RTOL = 1e-4
SCORE_RTOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def run_gpu(w: synth.Workload, seed=None, stream=None, greedy=False, shared_prefix_row=False):
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype, stream=stream,
                    shared_q=w.shared_q and not greedy, greedy=greedy,
                    shared_prefix_row=shared_prefix_row)
    out = v(w.p_logits, None if greedy else w.q_logits, w.drafts, temperature=w.temperature,
            seed=w.seed if seed is None else seed, temps=w.temps, scores=True, lse=True)
    status = bd.sdv_sync(v.ctx)
    res = {k: t.cpu().numpy() for k, t in out.items()}
    res["status"] = status
    res["plan"] = v.plan()
    v.close()
    return res


def run_oracle(w: synth.Workload, seqs=None, seed=None, greedy=False, lens=None):
    """The oracle on the whole batch in one call over all host threads (one
    thread per sequence), or on the listed sequences, each keeping its own b
    in the uniform keying."""
    import oracle
    p, q, d, t = synth.to_oracle_arrays(w, seqs)
    seed = w.seed if seed is None else seed
    nt = oracle.max_threads()
    if seqs is None:
        if greedy:
            return oracle.verify_greedy(p, d, t, seed, nthreads=nt, lens=lens)
        return oracle.verify(p, q, d, t, seed, nthreads=nt, lens=lens)
    outs = []
    for i, b in enumerate(seqs):
        ln = None if lens is None else lens[b:b + 1]
        if greedy:
            outs.append(oracle.verify_greedy(p[i:i + 1], d[i:i + 1], t[i:i + 1], seed, b0=b,
                                             nthreads=nt, lens=ln))
        else:
            outs.append(oracle.verify(p[i:i + 1], q[i:i + 1], d[i:i + 1], t[i:i + 1], seed, b0=b,
                                      nthreads=nt, lens=ln))
    return {k: np.concatenate([o[k] for o in outs]) for k in outs[0]}


BAND_NAMES = band_report.KINDS


def full_size_bounds(n: int) -> dict:
    """Band bounds of a full-size Qwen-vocabulary batch of n sequences.  The
    acceptance, selection and residual-mass kinds are rare (at most 2).  The
    CDF kind is not: a draw that lands on a token of mass below 1e-5 of the
    row's total lies wholly inside the band, and 152064-token rows hold many
    such tokens (their share of the draws is about sum_v min(p_v, 2e-5),
    around a tenth here), so it is bounded by a quarter of the trials."""
    return {"accept": 2, "select": 2, "resid": 2, "cdf": max(2, n // 4)}


def compare(gpu, orc, seqs=None, tag="", max_kind=None):
    """Assert parity on every listed sequence (all by default) and return the
    number of boundary-band trials as a band_report.BandCount (kinds and the
    band trials on which the GPU still agrees attached); the count is
    recorded for the run's summary.  Data-error trials must be -1 on both
    sides.  max_kind, when given, bounds the trials of each band kind: an int
    for every kind, or a dict by kind name."""
    seqs = list(range(len(orc["sel"]))) if seqs is None else list(seqs)
    n_band = n_agree = 0
    kinds = {}
    for i, b in enumerate(seqs):
        if orc["err"][i]:
            assert gpu["sel"][b] == -1 and gpu["accept_len"][b] == -1 and gpu["next_token"][b] == -1
            continue
        lg = gpu["lse"][b]
        lo = orc["lse"][i][..., :lg.shape[-1]]      # greedy mode has no q rows
        bad = np.abs(lg - lo) > LSE_RTOL * np.maximum(1.0, np.abs(lo))
        assert not bad.any(), "%s b=%d LSE mismatch %s vs %s" % (tag, b, lg[bad][:4], lo[bad][:4])
        so, sg = orc["scores"][i], gpu["scores"][b]
        assert np.all(np.abs(sg - so) <= SCORE_RTOL * np.abs(so) + 1e-6), \
            "%s b=%d scores %s vs %s" % (tag, b, sg, so)
        got = (int(gpu["sel"][b]), int(gpu["accept_len"][b]), int(gpu["next_token"][b]))
        exp = (int(orc["sel"][i]), int(orc["accept_len"][i]), int(orc["next_token"][i]))
        if orc["band"][i]:
            n_band += 1
            n_agree += got == exp
            for bit, name in BAND_NAMES.items():
                if orc["band"][i] & bit:
                    kinds[name] = kinds.get(name, 0) + 1
            continue
        assert got == exp, "%s b=%d (sel, L, token) gpu %s oracle %s" % (tag, b, got, exp)
    count = band_report.BandCount(n_band, checked=len(seqs), kinds=kinds, band_agree=n_agree,
                                  tag=tag)
    band_report.record(count)
    if n_band:
        print("%s: %d of %d trials in the boundary band %s, %d of them still equal"
              % (tag, n_band, len(seqs), kinds, n_agree))
    if max_kind is not None:
        for name, n in kinds.items():
            bound = max_kind[name] if isinstance(max_kind, dict) else max_kind
            assert n <= bound, "%s: %d trials in the %s band (bound %d)" % (tag, n, name, bound)
    return count


def _small(B, K, G, V, dtype=torch.bfloat16, T=1.0, seed=0, temps=None, identical=(),
           sigma=0.8, p_sigma=3.0, zipf=True):
    return synth.generate(B, K, G, V, dtype=dtype, p_sigma=p_sigma, zipf=zipf,
                          q_sigma=torch.full((B, K, G), sigma), identical=identical,
                          temperature=T, temps=temps, seed=seed, device="cuda")


# ---------------------------------------------------------------------------
# small shapes: full oracle comparison
# ---------------------------------------------------------------------------

def test_tiny_exact_workload():
    w = synth.workload(1, device="cuda")
    gpu, orc = run_gpu(w), run_oracle(w)
    assert gpu["status"] == bd.SDV_OK
    assert compare(gpu, orc, tag="tiny") == 0


def test_tiny_style_many_sequences_fp32():
    # many independent trials of the tiny exactness shape (V = 32, fp32)
    w = synth.generate(2048, 1, 4, 32, dtype=torch.float32, p_sigma=2.0, zipf=False,
                       q_sigma=torch.ones((2048, 1, 4)), seed=11, device="cuda")
    gpu, orc = run_gpu(w, seed=5), run_oracle(w, seed=5)
    nb = compare(gpu, orc, tag="tiny-many")
    assert nb <= 3, nb
    # the residual path and the bonus path both occur
    L = orc["accept_len"]
    assert (L < 4).any() and (L == 4).any()


@pytest.mark.parametrize("shape", [
    (4, 3, 5, 5000, 0.7),        # several chunks per row, ragged last chunk
    (3, 2, 3, 8, 1.0),           # one vector per row (bf16)
    (2, 4, 7, 12344, 1.3),       # V*2 = 16 * 1543: odd vector count
    (1, 1, 1, 152064, 1.0),      # gamma = 1
    (2, 2, 4, 3000, 5.0),        # high temperature: near-uniform rows
])
def test_small_shapes(shape):
    B, K, G, V, T = shape
    w = _small(B, K, G, V, T=T, seed=B * 1000 + V)
    gpu, orc = run_gpu(w, seed=7), run_oracle(w, seed=7)
    assert gpu["status"] == bd.SDV_OK
    assert compare(gpu, orc, tag=str(shape)) <= max(1, B // 100)


def test_very_low_temperature():
    """T = 0.05: near one-hot rows, most ratios within 1e-8 of 1, so many
    selections are genuine near-ties (boundary); every other trial matches."""
    B, K, G, V, T = 64, 6, 2, 2048, 0.05
    w = _small(B, K, G, V, T=T, seed=5 * 1000 + V)
    gpu, orc = run_gpu(w, seed=7), run_oracle(w, seed=7)
    assert gpu["status"] == bd.SDV_OK
    nb = compare(gpu, orc, tag="T=0.05")
    assert B - nb >= B // 4, "only %d of %d trials outside the band" % (B - nb, B)


def test_fp32_large_vocab():
    w = _small(3, 2, 3, 40000, dtype=torch.float32, T=0.9, seed=3)
    gpu, orc = run_gpu(w), run_oracle(w)
    assert compare(gpu, orc, tag="fp32") == 0


def test_single_stream_workload_full():
    w = synth.workload(2, device="cuda")
    gpu, orc = run_gpu(w), run_oracle(w)
    assert compare(gpu, orc, tag="single-stream") == 0


def test_self_selection_workload_full():
    w = synth.workload(3, device="cuda")
    gpu, orc = run_gpu(w), run_oracle(w)
    nb = compare(gpu, orc, tag="self-selection")
    assert nb <= 1
    assert len(set(orc["sel"].tolist())) > 1, "selection never moves off draft 0"


# ---------------------------------------------------------------------------
# full-size workloads: every sequence against the oracle
# ---------------------------------------------------------------------------

def test_serving_workload_full():
    w = synth.workload(4, device="cuda")
    gpu = run_gpu(w)
    assert gpu["status"] == bd.SDV_OK
    G = w.gamma
    ident = set(w.identical)
    assert len(ident) == 19
    for b in ident:                          # q == p: full acceptance, streak gamma, draft 0
        assert gpu["accept_len"][b] == G and gpu["sel"][b] == 0
        assert np.all(gpu["scores"][b] == G)
    orc = run_oracle(w)
    nb = compare(gpu, orc, tag="serving B64 K8 g16 (all 64)",
                 max_kind=full_size_bounds(64))
    assert nb <= 64 // 4 + 6
    del w
    torch.cuda.empty_cache()


def test_large_window_workload_full():
    w = synth.workload(5, device="cuda")
    gpu = run_gpu(w)
    assert gpu["status"] == bd.SDV_OK
    # the residual token carries residual mass: p > q at that id
    for b in range(w.B):
        L, k, x = int(gpu["accept_len"][b]), int(gpu["sel"][b]), int(gpu["next_token"][b])
        if L < w.gamma:
            lse = gpu["lse"][b, k]
            T = w.temps_list()[b]
            lp = float(w.p_logits[b, k, L, x]) / T - lse[L]
            lq = float(w.q_logits[b, k, L, x]) / T - lse[w.gamma + 1 + L]
            assert lp > lq - 1e-6
    orc = run_oracle(w)
    nb = compare(gpu, orc, tag="large-window B32 K16 g32 (all 32)",
                 max_kind=full_size_bounds(32))
    assert nb <= 32 // 4 + 6
    del w
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def test_identical_rows_everywhere():
    B, K, G, V = 6, 3, 4, 1000
    w = _small(B, K, G, V, identical=range(B), seed=21)
    gpu, orc = run_gpu(w), run_oracle(w)
    assert (gpu["accept_len"] == G).all() and (gpu["sel"] == 0).all()
    assert (gpu["scores"] == G).all()
    # the bonus draw may land on a low-mass token (CDF band); decisions
    # outside the band are compared exactly
    nb = compare(gpu, orc, tag="identical")
    assert nb < B and not (orc["band"] & ~2).any(), orc["band"]


def test_minus_inf_logits():
    """-inf entries carry no mass; q(x) = 0 accepts, p(x) = 0 < q(x) rejects."""
    B, K, G, V = 4, 2, 3, 512
    w = _small(B, K, G, V, seed=31)
    p, q, d = w.p_logits, w.q_logits, w.drafts
    ninf = float("-inf")
    p[:, :, :, 300:] = ninf                  # masked tail of the verifier rows
    q[:, :, :, 400:] = ninf
    d[0, 0, 0] = 350                         # p(x) = 0, q(x) > 0: reject at j = 0
    d[1, :, 1] = 450                         # q(x) = 0: accept at once
    p[2, :, :, 0] = ninf                     # a -inf in the middle of a row
    gpu, orc = run_gpu(w, seed=3), run_oracle(w, seed=3)
    assert compare(gpu, orc, tag="-inf") == 0
    # sequence 0 draft 0 has ratio 0 at j = 0: its score is 0
    assert gpu["scores"][0, 0] == 0.0
    assert (gpu["next_token"][gpu["next_token"] >= 0] < 300).all()


def test_one_token_rows():
    """Rows with a single finite entry: softmax is one-hot."""
    B, K, G, V = 3, 2, 2, 256
    w = _small(B, K, G, V, seed=41)
    w.p_logits.fill_(float("-inf"))
    w.q_logits.fill_(float("-inf"))
    w.p_logits[..., 7] = 1.5
    w.q_logits[..., 7] = -3.0
    w.drafts.fill_(7)
    gpu, orc = run_gpu(w), run_oracle(w)
    assert (gpu["accept_len"] == G).all() and (gpu["next_token"] == 7).all()
    assert compare(gpu, orc, tag="one-hot") == 0


def test_data_errors_reported():
    B, K, G, V = 4, 2, 3, 1024
    w = _small(B, K, G, V, seed=51)
    w.drafts[1, 1, 2] = V                          # draft id out of range
    w.p_logits[2, 0, 1, 10] = float("nan")         # NaN in a row
    temps = torch.tensor([1.0, 1.0, 1.0, -2.0], device="cuda")   # bad temperature
    w.temps = temps
    gpu = run_gpu(w)
    assert gpu["status"] == bd.SDV_ERR_DEVICE_DATA
    assert list(gpu["sel"][1:]) == [-1, -1, -1]
    assert list(gpu["next_token"][1:]) == [-1, -1, -1]
    orc = run_oracle(w)
    compare(gpu, orc, tag="errors")
    # status is cleared by sdv_sync: a clean step afterwards reports OK
    w2 = _small(B, K, G, V, seed=52)
    assert run_gpu(w2)["status"] == bd.SDV_OK


def test_argument_errors():
    w = _small(2, 2, 2, 64, seed=61)
    v = bd.Verifier(2, 2, 2, 64)
    out = {k: torch.empty(2, dtype=torch.int32, device="cuda") for k in ("sel", "accept_len", "next_token")}
    st = bd.sdv_verify(v.ctx, w.p_logits, w.q_logits, w.drafts, 0.0, 0, out["sel"],
                       out["accept_len"], out["next_token"])
    assert st == bd.SDV_ERR_ARG and "temperature" in bd.sdv_last_error(v.ctx)
    host = w.p_logits.cpu()
    st = bd.load().sdv_verify(v.ctx, host.data_ptr(), w.q_logits.data_ptr(), w.drafts.data_ptr(),
                              1.0, 0, out["sel"].data_ptr(), out["accept_len"].data_ptr(),
                              out["next_token"].data_ptr())
    assert st == bd.SDV_ERR_ARG and "device pointer" in bd.sdv_last_error(v.ctx)
    raw = torch.empty(w.p_logits.numel() + 1, dtype=torch.bfloat16, device="cuda")
    st = bd.load().sdv_verify(v.ctx, raw.data_ptr() + 2, w.q_logits.data_ptr(), w.drafts.data_ptr(),
                              1.0, 0, out["sel"].data_ptr(), out["accept_len"].data_ptr(),
                              out["next_token"].data_ptr())
    assert st == bd.SDV_ERR_ARG and "aligned" in bd.sdv_last_error(v.ctx)
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    v.close()


def test_deterministic_and_seeded():
    w = _small(16, 4, 8, 20000, seed=71)
    a, b2 = run_gpu(w, seed=9), run_gpu(w, seed=9)
    for k in ("sel", "accept_len", "next_token", "scores", "lse"):
        assert np.array_equal(a[k], b2[k]), k
    c = run_gpu(w, seed=10)
    assert np.array_equal(a["sel"], c["sel"]) and np.array_equal(a["scores"], c["scores"])
    assert not np.array_equal(a["next_token"], c["next_token"]) or \
        not np.array_equal(a["accept_len"], c["accept_len"])


def test_per_sequence_temperature_matches_scalar():
    B, K, G, V = 4, 2, 3, 4096
    w = _small(B, K, G, V, T=0.8, seed=81)
    scalar = run_gpu(w)
    w.temps = torch.full((B,), 0.8, device="cuda")
    per_seq = run_gpu(w)
    for k in ("sel", "accept_len", "next_token", "scores", "lse"):
        assert np.array_equal(scalar[k], per_seq[k]), k


def test_host_entry_point_matches_device():
    w = _small(8, 3, 6, 7000, seed=91)
    dev = run_gpu(w, seed=4)
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype)
    hp, hq = w.p_logits.cpu().pin_memory(), w.q_logits.cpu().pin_memory()
    hd = w.drafts.cpu().pin_memory()
    outs = [torch.empty(w.B, dtype=torch.int32).pin_memory() for _ in range(3)]
    for _ in range(2):
        st = bd.sdv_verify_host(v.ctx, hp, hq, hd, w.temperature, None, 4, *outs)
        assert st == bd.SDV_OK
        assert np.array_equal(outs[0].numpy(), dev["sel"])
        assert np.array_equal(outs[1].numpy(), dev["accept_len"])
        assert np.array_equal(outs[2].numpy(), dev["next_token"])
    v.close()


def test_side_stream():
    w = _small(4, 2, 3, 3000, seed=101)
    s = torch.cuda.Stream()
    ref = run_gpu(w)
    with torch.cuda.stream(s):
        got = run_gpu(w, stream=s)
    for k in ("sel", "accept_len", "next_token"):
        assert np.array_equal(ref[k], got[k])


# ---------------------------------------------------------------------------
# shared drafter marginals (q is [B, gamma, V], one row per position)
# ---------------------------------------------------------------------------

def test_shared_marginals_small():
    w = synth.generate_shared(6, 4, 5, 3000, q_sigma=torch.full((6, 5), 0.8), temperature=0.9,
                              seed=111, device="cuda")
    gpu, orc = run_gpu(w, seed=3), run_oracle(w, seed=3)
    assert gpu["status"] == bd.SDV_OK
    assert compare(gpu, orc, tag="shared") <= 1


def test_shared_marginals_equal_full_layout_bitwise():
    """The shared layout gives bit-identical outputs to the full layout with
    the marginal rows copied to every draft."""
    w = synth.generate_shared(4, 3, 6, 20000, temps=torch.tensor([0.6, 1.0, 1.3, 0.8]), seed=112,
                              device="cuda")
    shared = run_gpu(w, seed=5)
    full = synth.Workload(name="full", B=w.B, K=w.K, gamma=w.gamma, V=w.V, dtype=w.dtype,
                          p_logits=w.p_logits,
                          q_logits=w.q_logits[:, None].expand(w.B, w.K, w.gamma, w.V).contiguous(),
                          drafts=w.drafts, temperature=w.temperature, temps=w.temps, seed=w.seed)
    ref = run_gpu(full, seed=5)
    for k in ("sel", "accept_len", "next_token", "scores", "lse"):
        assert np.array_equal(shared[k], ref[k]), k


def test_shared_marginals_large_window_full():
    """The shared-marginal bench configuration at full size: every sequence
    against the oracle, and the shared prefix-row layout (what the bench line
    uses) bit-identical to reading every prefix row."""
    w = synth.workload_shared(device="cuda")
    gpu = run_gpu(w)
    assert gpu["status"] == bd.SDV_OK
    orc = run_oracle(w)
    nb = compare(gpu, orc, tag="shared-marginal B32 K16 g32 (all 32)",
                 max_kind=full_size_bounds(32))
    assert nb <= 32 // 4 + 6
    del orc
    pre = run_gpu(w, shared_prefix_row=True)
    for k in ("sel", "accept_len", "next_token", "scores", "lse"):
        assert np.array_equal(pre[k], gpu[k]), k
    del w
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# greedy acceptance (no drafter rows)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [
    (6, 4, 5, 3000, 0.9, torch.bfloat16),
    (512, 1, 4, 32, 1.0, torch.float32),       # many tiny-exact-style trials
    (3, 2, 7, 12344, 1.3, torch.bfloat16),
])
def test_greedy_small_shapes(shape):
    B, K, G, V, T, dt = shape
    w = _small(B, K, G, V, dtype=dt, T=T, seed=B * 7 + V, p_sigma=2.0 if dt == torch.float32 else 3.0,
               zipf=dt != torch.float32)
    gpu, orc = run_gpu(w, seed=9, greedy=True), run_oracle(w, seed=9, greedy=True)
    assert gpu["status"] == bd.SDV_OK
    assert gpu["lse"].shape == (B, K, G + 1)
    assert compare(gpu, orc, tag="greedy %s" % (shape,)) <= max(1, B // 100)
    # the rejected token is never its own replacement
    d = w.drafts.cpu().numpy()
    for b in range(B):
        L, k = int(gpu["accept_len"][b]), int(gpu["sel"][b])
        if L < G:
            assert gpu["next_token"][b] != d[b, k, L]


def test_greedy_large_window_full():
    w = synth.workload(5, device="cuda")
    w.q_logits = None                        # greedy acceptance reads no drafter rows
    torch.cuda.empty_cache()
    gpu = run_gpu(w, greedy=True)
    assert gpu["status"] == bd.SDV_OK
    orc = run_oracle(w, greedy=True)
    nb = compare(gpu, orc, tag="greedy large-window (all 32)",
                 max_kind=full_size_bounds(32))
    assert nb <= 32 // 4 + 6
    del w
    torch.cuda.empty_cache()


def _poison_prefix_rows(w):
    """A copy of w whose prefix rows (b, k > 0, 0) hold NaN: with the shared
    prefix-row layout they must not be read."""
    p = w.p_logits.clone()
    p[:, 1:, 0, :] = float("nan")
    return synth.Workload(name=w.name + " poisoned", B=w.B, K=w.K, gamma=w.gamma, V=w.V,
                          dtype=w.dtype, p_logits=p, q_logits=w.q_logits, drafts=w.drafts,
                          temperature=w.temperature, temps=w.temps, seed=w.seed,
                          shared_q=w.shared_q)


@pytest.mark.parametrize("greedy", [False, True])
def test_shared_prefix_row_reads_one_prefix_row(greedy):
    """With SDV_FLAG_SHARED_PREFIX_ROW the other drafts' prefix rows are never
    read (NaN there changes nothing) and the outputs equal, bit for bit, the
    full layout's on inputs whose prefix rows are identical."""
    w = synth.generate_shared(5, 4, 6, 12000, temps=torch.tensor([0.6, 1.0, 1.3, 0.8, 1.0]),
                              seed=113, device="cuda")
    assert torch.equal(w.p_logits[:, 1:, 0], w.p_logits[:, :1, 0].expand(-1, w.K - 1, -1))
    ref = run_gpu(w, seed=7, greedy=greedy)
    got = run_gpu(_poison_prefix_rows(w), seed=7, greedy=greedy, shared_prefix_row=True)
    assert got["status"] == bd.SDV_OK
    for k in ("sel", "accept_len", "next_token", "scores", "lse"):
        assert np.array_equal(got[k], ref[k]), k
    orc = run_oracle(w, seed=7, greedy=greedy)
    assert compare(got, orc, tag="prefix row") <= 1


def test_shared_prefix_row_with_full_q_layout():
    w = synth.workload(3, device="cuda", seed=3)
    p = w.p_logits.clone()
    p[:, 1:, 0] = p[:, :1, 0]
    w.p_logits = p
    ref = run_gpu(w)
    got = run_gpu(_poison_prefix_rows(w), shared_prefix_row=True)
    for k in ("sel", "accept_len", "next_token", "scores", "lse"):
        assert np.array_equal(got[k], ref[k]), k


def test_greedy_rejects_shared_q_combination():
    with pytest.raises(bd.SdvError):
        bd.Verifier(2, 2, 2, 64, shared_q=True, greedy=True)


def test_largest_select_shape_and_the_limit_beyond_it():
    """K * gamma near the select kernel's shared-memory limit (64 drafts of
    128 tokens: 164 KB of row statistics per sequence) against the oracle;
    one size up is refused at create time."""
    w = _small(2, 64, 128, 64, dtype=torch.float32, T=1.0, seed=41, zipf=False, p_sigma=1.5)
    gpu, orc = run_gpu(w, seed=2), run_oracle(w, seed=2)
    assert gpu["status"] == bd.SDV_OK
    assert compare(gpu, orc, tag="K64 g128") <= 1
    with pytest.raises(bd.SdvError):
        bd.Verifier(1, 128, 128, 64, torch.float32)
