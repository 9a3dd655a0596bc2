"""The row pass's row mode: one CTA per row and one partial per row, which the
planner picks for batches whose rows fill most of one wave of row CTAs (the
self-selection shape, B8 K4 gamma16 over a 152064-token vocabulary: 1 056
rows).  The plan is checked through sdv_plan; the outputs against the oracle
with per-sequence draft lengths (rows past a length are skipped by whole
CTAs) and with the shared prefix row (the replaced prefix rows too), and on
shapes that land in the same window with fp32 logits, greedy acceptance and
shared marginals.  The full batch without either is in test_gpu_parity, and
the allocation-free entry point on this shape in test_zz_no_alloc."""
import numpy as np
import pytest
import torch

from draft_verification_sdv_gb300 import binding as bd
from draft_verification_sdv_gb300 import synth
from test_gpu_parity import compare, full_size_bounds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def test_plan_picks_row_mode_for_one_wave():
    V = 152064
    v = bd.Verifier(8, 4, 16, V, torch.bfloat16)
    plan = v.plan()
    v.close()
    assert plan["chunks_per_row"] == 1 and plan["chunk_vectors"] == V // 8
    assert plan["rowpass_ctas"] == 8 * 4 * 33                 # one CTA per row
    big = bd.Verifier(32, 4, 16, V, torch.bfloat16)          # four times the rows: item mode
    plan = big.plan()
    big.close()
    assert plan["chunks_per_row"] > 1


def test_row_mode_with_lengths_and_shared_prefix_row():
    w = synth.workload(3, device="cuda", seed=43)
    # every draft's prefix row equal to draft 0's, so the shared-prefix-row
    # layout (which reads only draft 0's) and the oracle see the same rows
    w.p_logits[:, 1:, 0] = w.p_logits[:, :1, 0]
    lens = np.array([16, 0, 5, 16, 1, 9, 12, 16], np.int32)
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype, shared_prefix_row=True)
    assert v.plan()["chunks_per_row"] == 1
    dl = torch.as_tensor(lens, dtype=torch.int32, device="cuda")
    out = v(w.p_logits, w.q_logits, w.drafts, temperature=w.temperature, seed=5, temps=w.temps,
            scores=True, lse=True, draft_len=dl)
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    gpu = {k: t.cpu().numpy() for k, t in out.items()}
    v.close()
    import oracle
    p, q, d, t = synth.to_oracle_arrays(w)
    orc = oracle.verify(p, q, d, t, 5, lens=lens, nthreads=oracle.max_threads())
    compare(gpu, orc, tag="row mode, lengths + shared prefix row", max_kind=full_size_bounds(w.B))
    assert ((gpu["accept_len"] >= 0) & (gpu["accept_len"] <= lens)).all()
    # rows past a length are not read: their LSE entries are NaN
    for b in range(w.B):
        L = int(lens[b])
        assert np.isnan(gpu["lse"][b, :, L + 1:w.gamma + 1]).all()
        assert np.isfinite(gpu["lse"][b, :, :L + 1]).all()


def _oracle_compare(w, gpu, greedy=False, tag=""):
    import oracle
    p, q, d, t = synth.to_oracle_arrays(w)
    if greedy:
        orc = oracle.verify_greedy(p, d, t, w.seed, nthreads=oracle.max_threads())
    else:
        orc = oracle.verify(p, q, d, t, w.seed, nthreads=oracle.max_threads())
    compare(gpu, orc, tag=tag, max_kind=full_size_bounds(w.B))


def _run(w, greedy=False, shared_prefix_row=False):
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype, shared_q=w.shared_q and not greedy,
                    greedy=greedy, shared_prefix_row=shared_prefix_row)
    assert v.plan()["chunks_per_row"] == 1                   # row mode
    out = v(w.p_logits, None if greedy else w.q_logits, w.drafts, temperature=w.temperature,
            seed=w.seed, temps=w.temps, scores=True, lse=True)
    assert bd.sdv_sync(v.ctx) == bd.SDV_OK
    gpu = {k: t.cpu().numpy() for k, t in out.items()}
    v.close()
    return gpu


def test_row_mode_fp32_rows():
    """The fp32 row kernel: 1 056 rows of 8 192 fp32 logits."""
    w = synth.generate(8, 4, 16, 8192, dtype=torch.float32, q_sigma=torch.full((8, 4, 16), 0.8),
                       temps=torch.tensor([0.6, 1.0, 1.3, 0.8] * 2), seed=45, device="cuda")
    _oracle_compare(w, _run(w), tag="row mode fp32")


def test_row_mode_greedy():
    """Greedy acceptance (verifier rows only): 8 x 4 x 33 = 1 056 rows."""
    w = synth.generate(8, 4, 32, 8192, q_sigma=torch.full((8, 4, 32), 0.8), temperature=0.9,
                       seed=46, device="cuda")
    _oracle_compare(w, _run(w, greedy=True), greedy=True, tag="row mode greedy")


def test_row_mode_shared_marginals():
    """Shared marginals and the shared prefix row: 8 x 4 x 25 + 8 x 24 = 992 rows planned."""
    w = synth.generate_shared(8, 4, 24, 8192, q_sigma=torch.full((8, 24), 0.7),
                              temps=torch.tensor([0.7, 1.0] * 4), seed=47, device="cuda")
    _oracle_compare(w, _run(w, shared_prefix_row=True), tag="row mode shared marginals")
