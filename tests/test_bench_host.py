"""Host logic of bench.py, without a GPU: the algorithmic byte counts behind
the roofline (rows of each workload as the scope table states them, the
shared layouts, greedy acceptance, the re-read rows of the draw), the peak
lookup, and the traffic figures read from the committed ncu summaries."""
import json
import os
import sys
import types

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

V = 152064


def _w(B, K, G, V, dtype=torch.bfloat16, shared_q=False):
    return types.SimpleNamespace(B=B, K=K, gamma=G, V=V, dtype=dtype, shared_q=shared_q)


@pytest.mark.parametrize("shape,rows", [((1, 1, 4, 32, torch.float32), 9),
                                        ((1, 1, 8, V, torch.bfloat16), 17),
                                        ((8, 4, 16, V, torch.bfloat16), 1056),
                                        ((64, 8, 16, V, torch.bfloat16), 16896),
                                        ((32, 16, 32, V, torch.bfloat16), 33280)])
def test_rows_of_each_workload(shape, rows):
    B, K, G, v, dt = shape
    sb = bench.step_bytes(_w(B, K, G, v, dt), [G] * B)
    assert sb["rows"] == rows
    elt = 2 if dt == torch.bfloat16 else 4
    assert sb["k1"] == rows * v * elt
    # every sequence accepted everything: one bonus row each
    assert sb["reread_rows"] == B
    assert sb["total"] == sb["k1"] + B * v * elt + B * K * G * 4 + B * 12


def test_large_window_row_pass_bytes():
    assert bench.step_bytes(_w(32, 16, 32, V), [32] * 32)["k1"] == 10_121_379_840


def test_shared_layouts_greedy_and_the_draw():
    B, K, G, v = 2, 3, 4, 64
    w = _w(B, K, G, v, shared_q=True)
    # one prefix row per sequence, one marginal row per position
    assert bench.step_bytes(w, [G, G], shared_prefix_row=True)["rows"] == B * (K * G + 1) + B * G
    assert bench.step_bytes(w, [G, G])["rows"] == B * K * (G + 1) + B * G
    # greedy: no drafter rows, and a replacement reads one row
    g = bench.step_bytes(_w(B, K, G, v), [1, G], greedy=True)
    assert g["rows"] == B * K * (G + 1) and g["reread_rows"] == 2
    # a residual re-reads two rows, a bonus one
    assert bench.step_bytes(_w(B, K, G, v), [1, G])["reread_rows"] == 3


def test_measured_peak_lookup():
    peak, kind = bench.measured_peaks()
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            assert (peak, kind) == (float(json.load(f)["hbm_gbs"]), "measured")
    else:
        assert kind == "fallback"


@pytest.mark.parametrize("which", ["rowpass", "cps"])
def test_traffic_figures_of_the_committed_summaries(which):
    """A summary counts while its recorded source hash is that of the
    kernel's sources; its figure is then one 304 128-byte bf16 row plus a
    little (no re-reads)."""
    profile, sources = ((bench.TRAFFIC_PROFILE, bench.ROWPASS_SOURCES) if which == "rowpass"
                        else (bench.CPS_TRAFFIC_PROFILE, bench.CPS_SOURCES))
    t = bench.traffic_per_row(profile, sources)
    if t is None:
        pytest.skip("the summary predates the kernel's sources; the bench reports traffic null")
    assert V * 2 <= t <= 1.02 * V * 2
    # a different source hash is not taken
    assert bench.traffic_per_row(profile, sources[:1]) is None or len(sources) == 1


def _trial(sel, L, tok, band=0, err=0, lse=0.0, score=1.0):
    return dict(sel=sel, L=L, tok=tok, band=band, err=err, lse=lse, score=score)


def _as_arrays(trials, gpu_shift=None):
    import numpy as np
    n = len(trials)
    orc = {"sel": np.array([t["sel"] for t in trials]), "accept_len": np.array([t["L"] for t in trials]),
           "next_token": np.array([t["tok"] for t in trials]), "band": np.array([t["band"] for t in trials]),
           "err": np.array([t["err"] for t in trials]),
           "lse": np.array([[t["lse"], t["lse"]] for t in trials]),
           "scores": np.array([[t["score"]] for t in trials])}
    gpu = {k: orc[k].copy() for k in ("sel", "accept_len", "next_token")}
    gpu["lse"] = orc["lse"].astype(np.float32).copy()
    gpu["scores"] = orc["scores"].astype(np.float32).copy()
    for i in range(n):
        if orc["err"][i]:
            gpu["sel"][i] = gpu["accept_len"][i] = gpu["next_token"][i] = -1
    if gpu_shift:
        for i, k, dv in gpu_shift:
            gpu[k][i] += dv
    return gpu, orc


def test_parity_block_counts_mismatches_and_band_kinds():
    """The bench's parity block: a decision that differs outside the band is
    a mismatch; inside the band it is counted by kind (a trial may hold
    several) and as agreeing or not; data errors must be -1 on the GPU."""
    trials = [_trial(0, 3, 7), _trial(1, 0, 5), _trial(2, 4, 9, band=1 | 8), _trial(0, 2, 4, band=2),
              _trial(-1, -1, -1, err=1), _trial(3, 1, 11, band=4)]
    gpu, orc = _as_arrays(trials, gpu_shift=[(1, "next_token", 1), (3, "accept_len", 1)])
    p = bench.parity_block(gpu, orc)
    assert p["checked"] == 6 and p["data_errors"] == 1
    assert p["mismatches"] == 1                       # trial 1; trial 3 differs inside the band
    assert p["band_trials"] == 3 and p["band_agree"] == 2
    assert p["band"] == {"accept": 1, "cdf": 1, "select": 1, "resid": 1}
    assert p["lse_max_rel_err"] == 0.0 and p["score_max_rel_err"] == 0.0


def test_parity_block_flags_a_data_error_the_gpu_missed():
    trials = [_trial(-1, -1, -1, err=2), _trial(0, 1, 3)]
    gpu, orc = _as_arrays(trials)
    gpu["sel"][0] = 0                                  # the GPU did not report the bad row
    assert bench.parity_block(gpu, orc)["mismatches"] == 1
