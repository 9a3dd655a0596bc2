"""Parity of the causal-consistency path search (sdv_cps, through the C ABI)
with the fp64 oracle.

Bar: candidate ids and counts, lattice lengths, path ids and path counts
bit-exact, except sequences the oracle flags in its band (a cumulative mass
within 1e-5 of tau at a cut); candidate raw logits exact; candidate
log-probabilities and path scores within 1e-4 (absolute, relative for
scores).  The path order needs no band: the oracle ranks paths by fp64 sums
of raw logits and the kernel by fp64 sums of their differences to the best
path's, both exact for these logits, so they order paths alike."""
import numpy as np
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


def _host(q):
    q = q.detach().cpu().contiguous()
    if q.dtype == torch.bfloat16:
        return q.view(torch.int16).numpy().view(np.uint16)
    return q.numpy()


def run_both(q, temps, tau, mmax, beam, eos=-1):
    g = bd.sdv_cps(q, tau=tau, mmax=mmax, beam=beam, eos_id=eos,
                   temps=temps if torch.is_tensor(temps) else None,
                   temperature=1.0 if torch.is_tensor(temps) else float(temps))
    torch.cuda.synchronize()
    gpu = {k: v.cpu().numpy() for k, v in g.items()}
    import oracle
    t = temps.cpu().numpy() if torch.is_tensor(temps) else temps
    orc = oracle.cps(_host(q), t, tau, mmax, beam, eos_id=eos, nthreads=oracle.max_threads())
    return gpu, orc


def compare_cps(gpu, orc, tag="", q=None):
    B = gpu["npaths"].shape[0]
    n_band = 0
    for b in range(B):
        assert gpu["lat_len"][b] == orc["lat_len"][b], (tag, b)
        if orc["band"][b] & 1:
            n_band += 1
            continue
        assert np.array_equal(gpu["ncand"][b], orc["ncand"][b]), (tag, b)
        assert np.array_equal(gpu["cand_ids"][b], orc["cand_ids"][b]), (tag, b)
        lo, lg = orc["cand_logp"][b], gpu["cand_logp"][b]
        fin = np.isfinite(lo)
        assert np.array_equal(fin, np.isfinite(lg))
        assert np.all(np.abs(lg[fin] - lo[fin]) <= 1e-4), (tag, b)
        if q is not None:                  # raw logits of the candidates, exactly
            ids = gpu["cand_ids"][b]
            raw = np.where(ids >= 0, np.take_along_axis(q[b], np.maximum(ids, 0), axis=1), -np.inf)
            assert np.array_equal(gpu["cand_logit"][b], raw.astype(np.float32)), (tag, b)
        assert gpu["npaths"][b] == orc["npaths"][b], (tag, b)
        assert np.array_equal(gpu["paths"][b], orc["paths"][b]), (tag, b, gpu["paths"][b], orc["paths"][b])
        n = orc["npaths"][b]
        assert np.all(np.abs(gpu["path_logp"][b, :n] - orc["path_logp"][b, :n])
                      <= 1e-4 * (1 + np.abs(orc["path_logp"][b, :n])))
    return n_band


def _qf(q):
    return q.float().cpu().numpy()


@pytest.mark.parametrize("shape", [(4, 6, 3000, 0.8, 15, 3), (3, 5, 40000, 0.5, 8, 7),
                                   (2, 3, 64, 0.95, 16, 16), (5, 8, 5000, 0.0, 4, 2)])
def test_cps_small_shapes(shape):
    B, G, V, tau, mmax, beam = shape
    gen = torch.Generator(device="cuda")
    gen.manual_seed(B * 100 + G)
    q = (torch.randn((B, G, V), generator=gen, device="cuda") * 2.5).to(torch.bfloat16)
    gpu, orc = run_both(q, 0.9, tau, mmax, beam)
    assert compare_cps(gpu, orc, str(shape), _qf(q)) <= 1


def test_cps_fp32_ties_and_eos():
    B, G, V, eos = 4, 6, 512, 11
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    q = torch.randn((B, G, V), generator=gen, device="cuda")
    q[:, :, 100:104] = q[:, :, 100:101] + 3.0          # tied candidates
    q[1, 3, eos] = 20.0                                 # EOS ends sequence 1 at position 3
    q[1, :3, eos] = -20.0
    gpu, orc = run_both(q, torch.tensor([0.7, 1.0, 1.3, 2.0], device="cuda"), 0.8, 6, 4, eos=eos)
    assert compare_cps(gpu, orc, "fp32", _qf(q)) == 0
    assert gpu["lat_len"][1] == 4 and (gpu["paths"][1, :, 4:] == -1).all()


def test_cps_large_window_marginals():
    w = synth.workload_shared(B=8, device="cuda", seed=71)
    gpu, orc = run_both(w.q_logits, w.temps, 0.8, 15, 3)
    assert compare_cps(gpu, orc, "large-window", _qf(w.q_logits)) <= 1


def test_cps_paths_as_drafts_verify_end_to_end():
    """CPS paths are the K = beam drafts of a shared-marginal verification."""
    B, K, G, V = 6, 3, 8, 4000
    w = synth.generate_shared(B, K, G, V, q_sigma=torch.full((B, G), 0.6), temperature=1.0,
                              seed=72, device="cuda")
    cps = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=K)
    torch.cuda.synchronize()
    assert (cps["npaths"] == K).all() and (cps["lat_len"] == G).all()
    w.drafts = cps["paths"].contiguous()
    v = bd.Verifier(B, K, G, V, shared_q=True)
    out = v(w.p_logits, w.q_logits, w.drafts, temperature=1.0, seed=3, scores=True, lse=True)
    v.sync()
    import oracle
    p, q, d, t = synth.to_oracle_arrays(w)
    orc = oracle.verify(p, q, d, t, 3)
    gpu = {k: x.cpu().numpy() for k, x in out.items()}
    for b in range(B):
        if orc["band"][b]:
            continue
        assert (gpu["sel"][b], gpu["accept_len"][b], gpu["next_token"][b]) == \
            (orc["sel"][b], orc["accept_len"][b], orc["next_token"][b])
    v.close()


def test_cps_argument_errors():
    q = torch.zeros((2, 3, 64), dtype=torch.bfloat16, device="cuda")
    for kw in (dict(mmax=17), dict(beam=0), dict(tau=1.5), dict(eos_id=64)):
        with pytest.raises(bd.SdvError):
            bd.sdv_cps(q, **kw)


def test_cps_zero_probability_and_bad_rows():
    """-inf logits are never candidates; a row with NaN / +inf, or no finite
    logit, keeps none and its sequence has no path."""
    B, G, V = 4, 4, 1000
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    q = torch.randn((B, G, V), generator=gen, device="cuda")
    q[0, 1, :] = float("-inf")
    q[0, 1, torch.tensor([5, 77, 900])] = torch.tensor([1.0, 3.0, 2.0], device="cuda")
    q[1, 2, 10] = float("nan")
    q[2, 0, :] = float("-inf")
    q[3, 3, 999] = float("inf")
    for dt in (torch.float32, torch.bfloat16):
        gpu, orc = run_both(q.to(dt), 1.0, 0.9999, 15, 3)
        assert compare_cps(gpu, orc, str(dt), _qf(q.to(dt))) == 0
        assert list(gpu["cand_ids"][0, 1, :4]) == [77, 900, 5, -1]
        assert [gpu["npaths"][b] for b in range(B)] == [3, 0, 0, 0]


def test_cps_halves_equal_whole():
    """sdv_cps_prune then sdv_cps_beam gives exactly what sdv_cps gives; the
    pruned lattice before the EOS position is the final one."""
    B, G, V, eos = 3, 7, 5000, 17
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    q = (torch.randn((B, G, V), generator=gen, device="cuda") * 2.0).to(torch.bfloat16)
    q[:, :, eos] = -30.0
    q[1, 4, eos] = 30.0                                  # sequence 1 ends at position 4
    temps = torch.tensor([0.6, 1.0, 1.4], device="cuda")
    whole = bd.sdv_cps(q, 0.7, 10, 4, eos_id=eos, temps=temps)
    lat = bd.sdv_cps_prune(q, 0.7, 10, temps=temps)
    raw = {k: v.clone() for k, v in lat.items()}
    half = bd.sdv_cps_beam(lat, V, 4, eos_id=eos)
    torch.cuda.synchronize()
    for k in whole:
        assert torch.equal(whole[k], half[k]), k
    assert int(whole["lat_len"][1]) == 5
    assert torch.equal(raw["cand_ids"][1, :4], whole["cand_ids"][1, :4])
    assert int(raw["ncand"][1, 4]) >= 1 and int(whole["ncand"][1, 4]) == 1
    assert (whole["ncand"][1, 5:] == 0).all()


@pytest.mark.parametrize("beam", [3, 7])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_cps_exact_ties_on_a_coarse_grid(dt, beam):
    """Logits on a quarter grid: many paths tie exactly in their score; the
    order must be the tie rule's on both sides, not rounding's.  Beam 7 also
    takes paths with two and three deviations from the best path."""
    B, G, V = 6, 8, 2000
    gen = torch.Generator(device="cuda")
    gen.manual_seed(13)
    q = (torch.round(torch.randn((B, G, V), generator=gen, device="cuda") * 4) / 4 * 1.5).to(dt)
    gpu, orc = run_both(q, torch.tensor([0.6, 1.0, 1.0, 0.8, 1.3, 0.7], device="cuda"), 0.9, 12, beam)
    assert compare_cps(gpu, orc, "grid", _qf(q)) <= 1


def test_cps_four_warp_rows_full_size():
    """The bench's shape (1024 rows: one CTA of 4 warps per row) against the
    oracle on every sequence, and a smaller many-row case in full."""
    w = synth.workload_shared(B=32, device="cuda", seed=57)
    g = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=3, temps=w.temps)
    torch.cuda.synchronize()
    gpu = {k: v.cpu().numpy() for k, v in g.items()}
    import oracle
    orc = oracle.cps(_host(w.q_logits), w.temps.cpu().numpy(), 0.8, 15, 3,
                     nthreads=oracle.max_threads())
    assert compare_cps(gpu, orc, "full-size", _qf(w.q_logits)) <= 2
    del w, g
    torch.cuda.empty_cache()
    # 20 x 32 = 640 rows, all compared, bf16 and fp32
    gen = torch.Generator(device="cuda")
    gen.manual_seed(58)
    q32 = torch.randn((20, 32, 2000), generator=gen, device="cuda") * 2.0
    for q in (q32.to(torch.bfloat16), q32):
        gpu, orc = run_both(q, 0.8, 0.8, 15, 3)
        assert compare_cps(gpu, orc, "640 rows %s" % q.dtype, _qf(q)) <= 1


def test_cps_full_size_is_deterministic():
    """Every output of the path search, the row statistics included, is the
    same bit for bit on every run at the bench's size (152064-logit rows of
    many chunks per warp)."""
    w = synth.workload_shared(B=32, device="cuda", seed=59)
    runs = []
    for _ in range(3):
        o = bd.sdv_cps(w.q_logits, tau=0.8, mmax=15, beam=3, temps=w.temps, row_stat=True)
        torch.cuda.synchronize()
        runs.append({k: t.clone() for k, t in o.items()})
    for r in runs[1:]:
        for k in runs[0]:
            assert torch.equal(runs[0][k], r[k]), k
    del w, runs
    torch.cuda.empty_cache()


def test_cps_deterministic_and_argmax_path():
    gen = torch.Generator(device="cuda")
    gen.manual_seed(59)
    q = torch.randn((7, 9, 3000), generator=gen, device="cuda")
    a = bd.sdv_cps(q, tau=0.9, mmax=12, beam=5, temperature=0.7)
    b = bd.sdv_cps(q, tau=0.9, mmax=12, beam=5, temperature=0.7)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    # beam 1 keeps the most likely candidate at every position
    one = bd.sdv_cps(q, tau=0.9, mmax=12, beam=1, temperature=0.7)
    torch.cuda.synchronize()
    assert torch.equal(one["paths"][:, 0].long(), q.argmax(-1))


def test_cps_largest_lattice():
    """gamma 1024 positions, 16 candidates, beam 16 (the limits: 216 KB of
    shared memory for the beam, a frontier of up to 1 171 paths) against the
    oracle."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(60)
    q = (torch.randn((2, 1024, 256), generator=gen, device="cuda") * 0.7).to(torch.bfloat16)
    gpu, orc = run_both(q, 1.0, 0.999, 16, 16)
    assert compare_cps(gpu, orc, "g1024 w16", _qf(q)) <= 1
    assert (gpu["npaths"] == 16).all()
    with pytest.raises(bd.SdvError):
        bd.sdv_cps(torch.zeros((1, 1025, 64), dtype=torch.bfloat16, device="cuda"))


def _lattice_rows(spec, V, device="cuda"):
    """Marginal rows whose pruned lattice is exactly `spec`: spec[b][j] is the
    list of (token, logit) candidates of position j (at most 16, bf16-exact
    logits within one unit of each other); every other token gets logit -20.
    With tau 0.999 the cut falls after the last listed token: the mass left
    after it is below 1e-7 and the mass before it at most 0.98, both far from
    tau."""
    B, G = len(spec), len(spec[0])
    q = torch.full((B, G, V), -20.0)
    for b in range(B):
        for j in range(G):
            for tok, val in spec[b][j]:
                q[b, j, tok] = val
    return q.to(torch.bfloat16).to(device)


def _cands(n, grid, rng, V):
    toks = rng.choice(V, size=n, replace=False)
    return [(int(t), float(rng.choice(grid))) for t in toks]


@pytest.mark.parametrize("beam", [16, 3])
def test_cps_beam_frontier_edges(beam):
    """The best-first beam at its edges, against the oracle's beam: every
    path tied (only the lexicographic rule orders them), fewer paths than the
    beam (the frontier runs dry), a single path, a single position, sixteen
    candidates everywhere on a coarse grid (paths with up to four deviations),
    and 40 positions (two lanes' worth) with an EOS cut."""
    rng = np.random.default_rng(71 + beam)
    V, eos = 64, 7
    tied = [[(3, 0.0), (9, 0.0)]] * 5
    few = [[(1, 0.0), (2, 0.5)], [(3, 0.5), (4, 0.0)], [(5, 0.25), (6, 0.25)], [(8, 0.0)], [(10, 0.0)]]
    single = [[(11 + j, 0.0)] for j in range(5)]
    wide = [_cands(16, [0.0, 0.5, 1.0], rng, V) if j in (0, 4) else [(12, 0.0)] for j in range(5)]
    grid = [_cands(4, [0.0, 0.5, 1.0], rng, V) for _ in range(5)]
    q = _lattice_rows([tied, few, single, wide, grid], V)
    gpu, orc = run_both(q, 1.0, 0.999, 16, beam)
    assert compare_cps(gpu, orc, "edges", _qf(q)) == 0
    assert list(gpu["npaths"]) == [min(beam, 32), min(beam, 8), 1, beam, beam]

    one = _lattice_rows([[_cands(10, [0.0, 0.5], rng, V)]], V)      # gamma 1
    gpu, orc = run_both(one, 1.0, 0.999, 16, beam)
    assert compare_cps(gpu, orc, "gamma 1", _qf(one)) == 0
    assert gpu["npaths"][0] == min(beam, 10)

    G = 40
    deep = []
    for b in range(3):
        rows = []
        for j in range(G):
            n = 16 if b == 0 else int(rng.integers(1, 17))
            c = _cands(n, [0.0, 0.5, 1.0], rng, V)
            c = [(t, v) for t, v in c if t != eos] or [(eos + 1, 0.0)]
            rows.append(c)
        deep.append(rows)
    deep[2][35] = [(eos, 1.0), (20, 0.0)]                  # sequence 2 ends at position 35
    q = _lattice_rows(deep, V)
    gpu, orc = run_both(q, 1.0, 0.999, 16, beam, eos=eos)
    assert compare_cps(gpu, orc, "gamma 40", _qf(q)) == 0
    assert gpu["lat_len"][2] == 36 and gpu["lat_len"][0] == G
    assert (gpu["npaths"] == beam).all()
