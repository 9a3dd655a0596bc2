#!/usr/bin/env python3
"""Throughput of batched lossless draft verification with self-selection.

One step = one call of the whole path (row softmax statistics, ratios,
expected streaks, self-selection, acceptance scan, residual / bonus draw)
over one batch of the large-window workload: B = 32 sequences, K = 16
drafts, gamma = 32, V = 152064 (Qwen2.5 vocabulary), bf16 logits, drafter
noise rising from 0.3 to 2.0 across the window, per-sequence temperatures in
{0.6, 1.0}.  Inputs are synthetic, seeded, resident in HBM (10.1 GB, far
larger than the 129 MB L2, so no flush is needed between steps; smaller workloads
flush the L2 before every step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sdv|reference]

N > 1 runs under torchrun, one rank per GPU, each rank verifying its own batch
(sequences are independent: weak scaling, no collective on the data path).
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from draft_verification_sdv_gb300 import synth  # noqa: E402

METRIC = "verified draft-tokens/s and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
UNIT = "draft-tokens/s"
DEFAULT_WORKLOAD = 5
ROWPASS_SOURCES = ["k1_rowpass.cu", "sdv_device.cuh"]
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "rowpass_large-window.md")
CPS_SOURCES = ["k4_cps.cu", "sdv_device.cuh"]
CPS_TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "cps_prune_large-window.md")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["sdv", "reference"], default="sdv")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--cps", action="store_true",
                    help="time the causal-consistency path search on the large-window marginals")
    ap.add_argument("--decode-step", action="store_true",
                    help="time one whole decode step over one pass's marginals: path search, "
                         "verification of the paths at their lattice lengths, draft-length update")
    ap.add_argument("--greedy", action="store_true",
                    help="greedy acceptance: verifier rows only, no drafter rows")
    ap.add_argument("--shared-q", action="store_true",
                    help="drafts from one pass's marginals: q is [B, gamma, V] (large-window shape)")
    ap.add_argument("--batch", type=int, default=None,
                    help="shrink B of the workload (profiling captures only)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time the bench workload alone (no per_config block)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device: int):
        self.samples = []
        self.proc = None
        gid = None
        try:
            gid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            gid = vis.split(",")[device] if vis else str(device)
        self.gid = gid

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
               "-lms", "100", "-i", self.gid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.samples:
            if t0 - 0.15 <= ts <= t1 + 0.15:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = sorted({self.NAMES[i] for r in rows for i in range(4)
                          if r[2 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_sha(sources) -> str:
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "draft_verification_sdv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_per_row(profile: str = None, sources=None):
    """DRAM bytes per logit row of a kernel (default: the row pass) from its
    committed ncu summary, or None when that summary is absent or predates the
    kernel's sources."""
    profile = profile or TRAFFIC_PROFILE
    sources = sources or ROWPASS_SOURCES
    try:
        kv = {}
        with open(profile) as f:
            for line in f:
                if ":" in line and line.strip().startswith(("kernel_source_sha256", "dram_bytes_per_row")):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip().strip("`")
        if kv.get("kernel_source_sha256") != source_sha(sources):
            return None
        return float(kv["dram_bytes_per_row"])
    except Exception:
        return None


def step_bytes(w: synth.Workload, accept_len, greedy: bool = False,
               shared_prefix_row: bool = False) -> dict:
    """Algorithmic bytes of one step: every logit row read once (one prefix
    row per sequence when the drafts share it), the re-read rows of the draw
    (two for a residual, one for a bonus or a greedy replacement), drafts,
    outputs."""
    elt = 2 if w.dtype == torch.bfloat16 else 4
    q_rows = 0 if greedy else (w.B if w.shared_q else w.B * w.K) * w.gamma
    p_rows = w.B * (w.K * w.gamma + 1) if shared_prefix_row else w.B * w.K * (w.gamma + 1)
    rows = p_rows + q_rows
    reread = sum(2 if int(L) < w.gamma and not greedy else 1 for L in accept_len)
    k1 = elt * w.V * rows
    total = k1 + elt * w.V * reread + w.B * w.K * w.gamma * 4 + w.B * 12
    return {"rows": rows, "k1": k1, "total": total, "reread_rows": reread}


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def measure_verify(bd, w: synth.Workload, args, stream, greedy: bool = False,
                   prefix_row: bool = False, world: int = 1, steps: int = None) -> dict:
    """Time `steps` verification steps of workload w on `stream` (CUDA events),
    then a second pass with per-kernel events.  Inputs smaller than twice the
    L2 would stay cached from one step to the next: then the L2 is flushed (a
    write larger than it) before every step, outside the timed region, and
    each step is timed alone."""
    dev = w.p_logits.device
    steps = args.steps if steps is None else steps
    # the inputs were made on torch's current stream; the steps run on
    # `stream` (non-blocking): order them after the inputs
    stream.wait_stream(torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    v = bd.Verifier(w.B, w.K, w.gamma, w.V, w.dtype, stream=stream, shared_q=w.shared_q,
                    greedy=greedy, shared_prefix_row=prefix_row)
    out = None

    def step():
        nonlocal out
        out = v(w.p_logits, None if greedy else w.q_logits, w.drafts, temperature=w.temperature,
                seed=w.seed, temps=w.temps, out=out)

    for _ in range(max(args.warmup, 3) if args.warmup > 0 else 0):
        step()
    v.sync()
    torch.cuda.synchronize()
    barrier(world)
    sb0 = step_bytes(w, [w.gamma] * w.B, greedy=greedy, shared_prefix_row=prefix_row)
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)
    flush_buf = None
    if sb0["k1"] < 2 * l2_bytes:
        flush_buf = torch.empty(max(2 * l2_bytes, 256 << 20) // 4, dtype=torch.int32, device=dev)

    def flush():
        if flush_buf is not None:
            with torch.cuda.stream(stream):
                flush_buf.zero_()

    torch.cuda.synchronize()
    barrier(world)
    t0 = time.time()
    if flush_buf is None:
        # K steps back to back on the context's stream, nothing between the
        # kernels (the select and sample kernels launch as programmatic
        # dependents of the kernel before them).
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms_total = ev0.elapsed_time(ev1)
    else:
        pairs = []
        for _ in range(steps):
            flush()
            e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e_a.record(stream)
            step()
            e_b.record(stream)
            pairs.append((e_a, e_b))
        torch.cuda.synchronize()
        ms_total = sum(e_a.elapsed_time(e_b) for e_a, e_b in pairs)
    t1 = time.time()
    barrier(world)
    # Second pass of K steps with CUDA events around each kernel (the events
    # serialise the kernels): per-kernel durations for the roofline.
    bd.sdv_profile_enable(v.ctx, True)
    for _ in range(steps):
        flush()
        step()
    torch.cuda.synchronize()
    bd.sdv_profile_enable(v.ctx, False)
    v.sync()
    ms_kernels, nprof = bd.sdv_profile_read(v.ctx)
    accept_len = out["accept_len"].cpu().tolist()
    l2 = ("inputs %.2f GB > L2 (%d MB): no flush" % (sb0["k1"] / 1e9, l2_bytes >> 20)
          if flush_buf is None else
          "inputs %.4f GB < 2x L2 (%d MB): L2 flushed by a %d MB write before every step, "
          "outside the timed region; each step timed alone"
          % (sb0["k1"] / 1e9, l2_bytes >> 20, flush_buf.numel() * 4 >> 20))
    del flush_buf
    return {"verifier": v, "out": out, "ms_total": ms_total, "steps": steps, "t0": t0, "t1": t1,
            "ms_kernels": ms_kernels, "nprof": nprof, "accept_len": accept_len, "l2": l2,
            "flushed": sb0["k1"] < 2 * l2_bytes}


def run_sdv(args, rank, world, local):
    from draft_verification_sdv_gb300 import binding as bd
    bd.load(build=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    if args.shared_q:
        w = synth.workload_shared(B=args.batch or 32, device=dev, seed=55 + 1000 * rank)
    else:
        w = synth.workload(args.workload, device=dev, seed=args.workload + 1000 * rank, B=args.batch)
    stream = torch.cuda.Stream(device=dev)
    # drafts from one pass's marginals also share the prefix row (j = 0)
    prefix_row = bool(w.shared_q)
    if args.greedy:
        w.q_logits = None
        torch.cuda.empty_cache()

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.25)
    m = measure_verify(bd, w, args, stream, greedy=args.greedy, prefix_row=prefix_row, world=world)
    v, out = m["verifier"], m["out"]
    ms_kernels, nprof, accept_len = m["ms_kernels"], m["nprof"], m["accept_len"]
    ms_max = max_over_ranks(m["ms_total"], world)
    tokens_per_step = w.B * w.K * w.gamma
    value = world * tokens_per_step * args.steps / (ms_max / 1e3)
    ms_step = ms_max / args.steps
    sb = step_bytes(w, accept_len, greedy=args.greedy, shared_prefix_row=prefix_row)
    peak, peak_kind = measured_peaks()
    k1_gbs = sb["k1"] / (ms_kernels[0] * 1e-3) / 1e9 if ms_kernels[0] > 0 else None
    step_gbs = sb["total"] / (ms_step * 1e-3) / 1e9
    tpr = traffic_per_row()
    roofline = {
        "bound": "hbm",
        "kernel": "rowpass_kernel (online softmax statistics of every logit row)",
        "achieved": round(k1_gbs, 1) if k1_gbs else None,
        "peak": peak,
        "peak_kind": peak_kind,
        "unit": "GB/s",
        "frac": round(k1_gbs / peak, 4) if k1_gbs else None,
        "traffic": round(tpr * sb["rows"]) if tpr else None,
        "algorithmic_bytes_per_launch": sb["k1"],
        "ms_per_launch": round(ms_kernels[0], 5),
    }
    result = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "input_dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded logits and drafts; no model weights)",
        "config": {"workload": w.name, "B": w.B, "K": w.K, "gamma": w.gamma, "V": w.V,
                   "q_layout": ("none (greedy acceptance)" if args.greedy else
                                "[B,gamma,V] shared by the K drafts" if w.shared_q else "[B,K,gamma,V]"),
                   "prefix_row": "one per sequence" if prefix_row else "one per draft",
                   "temperatures": "per-sequence {0.6, 1.0}" if w.temps is not None else w.temperature,
                   "l2": m["l2"],
                   "parallelism": "replicas (one batch per GPU)" if world > 1 else "1 GPU"},
        "committed_tokens_per_s": world * sum(int(L) + 1 for L in accept_len) * args.steps / (ms_max / 1e3),
        "hbm": {"step_gbs": round(step_gbs, 1), "frac": round(step_gbs / peak, 4),
                "bytes_per_step": sb["total"], "reread_rows": sb["reread_rows"]},
        "kernel_ms": {"rowpass": ms_kernels[0], "select": ms_kernels[1], "sample": ms_kernels[2],
                      "steps": nprof, "how": "second pass of the same steps, CUDA events around "
                                               "each kernel on the context stream"},
        "roofline": roofline,
        "gpu_launches": 3 * args.steps,      # in the timed region (row pass, select, sample)
        "clocks": clocks.summary(m["t0"], m["t1"]),
    }

    # End to end through the host-buffer entry point: inputs copied from pinned
    # host memory each step, outputs read back.
    if not args.no_e2e:
        hp = torch.empty(w.p_logits.shape, dtype=w.dtype, pin_memory=True)
        hp.copy_(w.p_logits)
        hq = None
        if w.q_logits is not None:
            hq = torch.empty(w.q_logits.shape, dtype=w.dtype, pin_memory=True)
            hq.copy_(w.q_logits)
        hd = w.drafts.cpu().pin_memory()
        ht = w.temps.cpu().pin_memory() if w.temps is not None else None
        outs = [torch.empty(w.B, dtype=torch.int32).pin_memory() for _ in range(3)]
        st = bd.sdv_verify_host(v.ctx, hp, hq, hd, w.temperature, ht, w.seed, *outs)
        assert st == bd.SDV_OK, bd.sdv_last_error(v.ctx)
        barrier(world)
        te0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            st = bd.sdv_verify_host(v.ctx, hp, hq, hd, w.temperature, ht, w.seed, *outs)
            assert st == bd.SDV_OK, bd.sdv_last_error(v.ctx)
        te = time.perf_counter() - te0
        te = max_over_ranks(te, world)
        h2d = hp.numel() * hp.element_size() + (hq.numel() * hq.element_size() if hq is not None else 0) + \
            hd.numel() * 4 + (ht.numel() * 4 if ht is not None else 0)
        result["e2e"] = {"value": world * tokens_per_step * args.e2e_steps / te, "unit": UNIT,
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 3 * w.B * 4,
                         "steps": args.e2e_steps, "ms_per_step": te * 1e3 / args.e2e_steps}
        del hp, hq

    # The outputs of the timed step again, with scores and row LSE, for the
    # parity check of the cpu_baseline leg.
    gpu = v(w.p_logits, None if args.greedy else w.q_logits, w.drafts, temperature=w.temperature,
            seed=w.seed, temps=w.temps, scores=True, lse=True)
    v.sync()
    gpu = {k: t.cpu().numpy() for k, t in gpu.items()}
    v.close()

    # The oracle as it stands on the host cores, bounded sample (rank 0, N = 1),
    # and its parity with the GPU's outputs on the same sequences.
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.greedy:
        result["cpu_baseline"], result["parity"] = cpu_baseline(w, gpu)

    # The other workloads, timed in the same run (single-GPU line only).
    if (rank == 0 and world == 1 and not args.no_per_config and not args.greedy and
            not args.shared_q and args.batch is None and args.workload == DEFAULT_WORKLOAD):
        del w
        torch.cuda.empty_cache()
        result["per_config"] = per_config(bd, args, stream, clocks, peak, peak_kind)
    time.sleep(0.2)
    clocks.stop()
    return result


def per_config(bd, args, stream, clocks, peak, peak_kind) -> dict:
    """Workloads 1-4 (the tiny exact case and the single stream as latencies
    with the L2 flushed before every step; the self-selection sweep and the
    serving batch as throughput), the whole decode step and the path search,
    each timed as its own line would time it, with the clocks of its window."""
    dev = torch.device("cuda", torch.cuda.current_device())
    res = {}
    for idx in (1, 2, 3, 4):
        w = synth.workload(idx, device=dev, seed=idx)
        m = measure_verify(bd, w, args, stream)
        m["verifier"].close()
        ms = m["ms_total"] / m["steps"]
        sb = step_bytes(w, m["accept_len"])
        k1 = m["ms_kernels"][0]
        e = {"workload": w.name, "ms_per_step": ms,
             "draft_tokens_per_s": w.B * w.K * w.gamma / (ms * 1e-3),
             "kernel_ms": {"rowpass": k1, "select": m["ms_kernels"][1],
                           "sample": m["ms_kernels"][2]},
             "l2": m["l2"], "clocks": clocks.summary(m["t0"], m["t1"])}
        if not m["flushed"]:
            rp = sb["k1"] / (k1 * 1e-3) / 1e9
            st = sb["total"] / (ms * 1e-3) / 1e9
            e.update({"rowpass_gbs": round(rp, 1), "rowpass_frac": round(rp / peak, 4),
                      "step_gbs": round(st, 1), "step_frac": round(st / peak, 4),
                      "peak": peak, "peak_kind": peak_kind})
        else:
            e["latency_us"] = round(ms * 1e3, 2)
        res[str(idx)] = e
        del w, m
        torch.cuda.empty_cache()
    ds = run_decode_step(args, 0, 1, bd=bd, clocks=clocks)
    res["decode_step"] = {"workload": ds["config"]["workload"], "ms_per_step": ds["ms_per_step"],
                          "sequence_steps_per_s": ds["value"], "step_gbs": ds["hbm"]["step_gbs"],
                          "step_frac": ds["hbm"]["frac"], "peak_kind": ds["hbm"]["peak_kind"],
                          "clocks": ds["clocks"]}
    torch.cuda.empty_cache()
    cps_args = argparse.Namespace(**vars(args))
    cps_args.no_e2e = True
    cps_args.no_cpu_baseline = True
    cp = run_cps(cps_args, 0, 1, bd=bd, clocks=clocks)
    res["path_search"] = {"workload": cp["config"]["workload"], "ms_per_step": cp["ms_per_step"],
                          "rows_per_s": cp["value"], "kernel_ms": cp["kernel_ms"],
                          "prune_gbs": cp["roofline"]["achieved"], "prune_frac": cp["roofline"]["frac"],
                          "clocks": cp["clocks"]}
    torch.cuda.empty_cache()
    return res


def run_cps(args, rank, world, bd=None, clocks=None):
    """Path search over the drafter marginals of the large-window shape
    (B 32, gamma 32, V 152064 bf16, per-sequence temperatures): beam 3, at most
    15 candidates, mass 0.8.  One step = sdv_cps (pruning of every row, then
    the beam).  The q rows (311 MB) exceed the L2, so no flush is needed."""
    if bd is None:
        from draft_verification_sdv_gb300 import binding as bd
        bd.load(build=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    w = synth.workload_shared(B=args.batch or 32, device=dev, seed=55 + 1000 * rank)
    q, temps = w.q_logits, w.temps
    del w
    torch.cuda.empty_cache()
    B, G, V = q.shape
    tau, mmax, beam = 0.8, 15, 3
    stream = torch.cuda.current_stream(dev)
    out = bd.sdv_cps(q, tau, mmax, beam, temps=temps)

    def step():
        bd.sdv_cps(q, tau, mmax, beam, temps=temps, out=out)

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    barrier(world)
    own_clocks = clocks is None
    if own_clocks:
        clocks = ClockSampler(dev.index)
        clocks.start()
        time.sleep(0.25)
    barrier(world)
    t0 = time.time()
    ms = timed(step, args.steps)
    t1 = time.time()
    ms = max_over_ranks(ms, world)
    # the two kernels timed alone, same events on the launching stream
    lat = {k: out[k] for k in ("cand_ids", "cand_logp", "cand_logit", "ncand")}
    ms_prune = timed(lambda: bd.sdv_cps_prune(q, tau, mmax, temps=temps, out=lat), args.steps)
    paths_out = dict(out)
    ms_beam = timed(lambda: bd.sdv_cps_beam(lat, V, beam, out=paths_out), args.steps)
    if own_clocks:
        time.sleep(0.2)
        clocks.stop()
    row_bytes = q.numel() * q.element_size()
    peak, kind = measured_peaks()
    gbs = row_bytes / (ms_prune * 1e-3) / 1e9
    tpr = traffic_per_row(CPS_TRAFFIC_PROFILE, CPS_SOURCES)
    res = {"metric": "drafter rows pruned and beam-searched per second (causal-consistency path search)",
           "value": world * B * G / (ms * 1e-3), "unit": "rows/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "input_dtype": "bf16", "data": "synthetic drafter marginals (seeded; no model weights)",
           "config": {"workload": "large-window marginals B%d gamma%d V%d bf16" % (B, G, V),
                      "beam": beam, "mmax": mmax, "tau": tau,
                      "temperatures": "per-sequence {0.6, 1.0}",
                      "l2": "inputs %.2f GB > L2 (%d MB): no flush" % (row_bytes / 1e9, l2_mb(dev)),
                      "parallelism": "replicas (one batch per GPU)" if world > 1 else "1 GPU"},
           "kernel_ms": {"prune": ms_prune, "beam": ms_beam,
                         "how": "each half timed alone over the same number of steps"},
           "roofline": {"bound": "hbm", "kernel": "cps_prune_kernel (one streaming pass per row)",
                        "achieved": round(gbs, 1), "peak": peak, "peak_kind": kind,
                        "unit": "GB/s", "frac": round(gbs / peak, 4),
                        "traffic": round(tpr * B * G) if tpr else None,
                        "algorithmic_bytes_per_launch": row_bytes,
                        "ms_per_launch": round(ms_prune, 5)},
           "gpu_launches": 2 * args.steps,
           "clocks": clocks.summary(t0, t1)}
    if not args.no_e2e:
        # host marginals in pinned memory, copied in each step; paths read back
        hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        hq.copy_(q)
        ht = temps.cpu().pin_memory()
        dq, dt_ = torch.empty_like(q), torch.empty_like(temps)
        hp = torch.empty((B, beam, G), dtype=torch.int32, pin_memory=True)
        hs = torch.empty((B, beam), dtype=torch.float32, pin_memory=True)
        hn = torch.empty((B,), dtype=torch.int32, pin_memory=True)

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            dt_.copy_(ht, non_blocking=True)
            bd.sdv_cps(dq, tau, mmax, beam, temps=dt_, out=out)
            hp.copy_(out["paths"], non_blocking=True)
            hs.copy_(out["path_logp"], non_blocking=True)
            hn.copy_(out["npaths"], non_blocking=True)
            torch.cuda.current_stream().synchronize()

        e2e_step()
        barrier(world)
        te0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        te = max_over_ranks(time.perf_counter() - te0, world)
        res["e2e"] = {"value": world * B * G * args.e2e_steps / te, "unit": "rows/s",
                      "h2d_bytes_per_step": row_bytes + ht.numel() * 4,
                      "d2h_bytes_per_step": hp.numel() * 4 + hs.numel() * 4 + hn.numel() * 4,
                      "steps": args.e2e_steps, "ms_per_step": te * 1e3 / args.e2e_steps}
        del hq, dq
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        S = max(1, min(os.cpu_count() or 1, B, 8))
        hq = q[:S].cpu()
        hq = hq.view(torch.int16).numpy().view("uint16") if q.dtype == torch.bfloat16 else hq.numpy()
        nt = min(S, oracle.max_threads()) if oracle.max_threads() > 1 else 1
        c0 = time.perf_counter()
        oracle.cps(hq, temps[:S].cpu().numpy(), tau, mmax, beam, nthreads=nt)
        dtc = time.perf_counter() - c0
        res["cpu_baseline"] = {"value": S * G / dtc, "unit": "rows/s", "cores": nt, "kind": "oracle",
                               "sample": "first %d of %d sequences (%d rows), one thread per "
                                         "sequence (%.1f s wall)" % (S, B, S * G, dtc)}
    return res


ARM_PARTS = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1",
             "0xd49": "Arm Neoverse-N2"}


def run_decode_step(args, rank, world, bd=None, clocks=None):
    """One decode step of a diffusion drafter's pass, end to end on the GPU:
    the path search over the marginals q [B, gamma, V] (beam 3, 15
    candidates, mass 0.8, EOS cut), verification of the beam's K = 3 paths at
    their lattice lengths (shared marginals, shared prefix row), and the
    draft-length update from the lattice and accepted lengths.  The path
    search hands the marginal rows' softmax statistics to the verification,
    which therefore streams only the verifier rows.  Large-window shape: B 32,
    gamma 32, V 152064 bf16, per-sequence temperatures.

    The three run in order on one stream, as in a decode loop: the verifier
    rows are the verifier's distributions at the drafted paths' positions, so
    they exist only once the search has produced the paths (here they are
    synthesised up front, standing in for the verifier's forward pass), and
    the next step's search waits for this step's draft-length update."""
    if bd is None:
        from draft_verification_sdv_gb300 import binding as bd
        bd.load(build=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    B, K, G, V = args.batch or 32, 3, 32, synth.QWEN_VOCAB
    g = torch.Generator(device="cpu")
    g.manual_seed(10_055 + 1000 * rank)
    sj = 0.3 + 1.7 * torch.arange(G, dtype=torch.float32) / (G - 1)
    temps = torch.where(torch.rand((B,), generator=g) < 0.5, torch.tensor(0.6), torch.tensor(1.0))
    w = synth.generate_shared(B, K, G, V, q_sigma=sj.expand(B, G).clone(), temps=temps,
                              seed=55 + 1000 * rank, device=dev)
    eos = 151643                                   # the Qwen2.5 end-of-text id
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    v = bd.Verifier(B, K, G, V, w.dtype, shared_q=True, shared_prefix_row=True, stream=stream)
    ctl = bd.DraftLengthController(B, G, window=2, kmin=4, kmax=G, up=2, down=1, device=dev)
    cps = bd.sdv_cps(w.q_logits, 0.8, 15, K, eos_id=eos, temps=w.temps, row_stat=True, stream=stream)
    torch.cuda.synchronize(dev)
    out = None

    def step(i):
        nonlocal out
        bd.sdv_cps(w.q_logits, 0.8, 15, K, eos_id=eos, temps=w.temps, out=cps, row_stat=True,
                   stream=stream)
        out = v(w.p_logits, w.q_logits, cps["paths"], seed=i, temps=w.temps, out=out,
                draft_len=cps["lat_len"], q_stat=cps["row_stat"])
        ctl.step(cps["lat_len"], out["accept_len"], stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    v.sync()
    barrier(world)
    own_clocks = clocks is None
    if own_clocks:
        clocks = ClockSampler(dev.index)
        clocks.start()
        time.sleep(0.25)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if own_clocks:
        time.sleep(0.2)
        clocks.stop()
    v.sync()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    lat = cps["lat_len"].cpu().numpy()
    acc = out["accept_len"].cpu().numpy()
    elt = 2
    rows = B * G + sum(1 + K * int(L) for L in lat)                            # q once, p
    rows += sum(2 if int(a) < int(L) else 1 for a, L in zip(acc, lat))         # the draw
    gbs = rows * V * elt / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    committed = int(sum(int(a) + 1 for a in acc))
    v.close()
    l2_note = "inputs %.2f GB > L2 (%d MB): no flush" % (
        (w.p_logits.numel() + w.q_logits.numel()) * elt / 1e9, l2_mb(dev))
    del w, cps, out
    return {"metric": "decode steps per second (path search + verification + draft-length "
                      "update), sequences x steps / s",
            "value": world * B / (ms * 1e-3), "unit": "sequence-steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "input_dtype": "bf16", "data": "synthetic marginals and verifier rows (seeded)",
            "config": {"workload": "large-window marginals B%d K%d gamma%d V%d bf16" % (B, K, G, V),
                       "beam": K, "mmax": 15, "tau": 0.8, "eos_id": eos,
                       "marginal_rows": "streamed once (the path search's statistics feed "
                                        "the verification)",
                       "order": "one stream: path search, verification of its paths, "
                                "draft-length update",
                       "lattice_len_mean": float(lat.mean()),
                       "l2": l2_note},
            "committed_tokens_per_s": world * committed / (ms * 1e-3),
            "hbm": {"step_gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "peak": peak,
                    "peak_kind": kind, "rows_per_step": rows},
            "gpu_launches": 6 * args.steps,
            "clocks": clocks.summary(t0, t1)}


def l2_mb(dev) -> int:
    return getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20) >> 20


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                low = line.lower()
                if low.startswith("model name"):
                    return line.split(":", 1)[1].strip()
                if low.startswith("cpu part"):
                    part = line.split(":", 1)[1].strip()
                    return ARM_PARTS.get(part, "Arm CPU part " + part)
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


BAND_KINDS = {1: "accept", 2: "cdf", 4: "select", 8: "resid"}


def parity_block(gpu: dict, orc: dict) -> dict:
    """The GPU's outputs against the oracle's on the same sequences: decisions
    (selected draft, accepted length, emitted token) must be equal outside the
    oracle's 1e-5 boundary band; band trials are counted by kind, with how
    many still agree; row LSE and streak scores within 1e-4 relative."""
    import numpy as np
    n = len(orc["sel"])
    mism, band, agree, errs = 0, 0, 0, 0
    kinds = {name: 0 for name in BAND_KINDS.values()}
    lse_err = score_err = 0.0
    for b in range(n):
        got = (int(gpu["sel"][b]), int(gpu["accept_len"][b]), int(gpu["next_token"][b]))
        if orc["err"][b]:
            errs += 1
            mism += got != (-1, -1, -1)
            continue
        exp = (int(orc["sel"][b]), int(orc["accept_len"][b]), int(orc["next_token"][b]))
        lo = orc["lse"][b][..., :gpu["lse"][b].shape[-1]]
        lse_err = max(lse_err, float(np.max(np.abs(gpu["lse"][b] - lo) / np.maximum(1.0, np.abs(lo)))))
        so = orc["scores"][b]
        score_err = max(score_err, float(np.max(np.abs(gpu["scores"][b] - so) /
                                                np.maximum(np.abs(so), 1e-2))))
        if orc["band"][b]:
            band += 1
            agree += got == exp
            for bit, name in BAND_KINDS.items():
                if orc["band"][b] & bit:
                    kinds[name] += 1
            continue
        mism += got != exp
    return {"checked": n, "mismatches": mism, "band_trials": band, "band": kinds,
            "band_agree": agree, "data_errors": errs, "lse_max_rel_err": lse_err,
            "score_max_rel_err": score_err,
            "bar": "sel, accept_len, next_token equal outside the 1e-5 boundary band; "
                   "LSE and scores within 1e-4 relative"}


def cpu_baseline(w: synth.Workload, gpu: dict = None):
    """The oracle on every sequence of the batch, one host thread per sequence
    (its time is the CPU baseline), then its single-thread rate on the first
    sequence; with the GPU's outputs of the same step, also the parity block."""
    import oracle
    cores = os.cpu_count() or 1
    p, q, d, t = synth.to_oracle_arrays(w)
    nt = min(w.B, oracle.max_threads()) if oracle.max_threads() > 1 else 1
    t0 = time.perf_counter()
    orc = oracle.verify(p, q, d, t, w.seed, nthreads=nt)
    dt = time.perf_counter() - t0
    # the same oracle on one thread, first sequence only
    t1 = time.perf_counter()
    oracle.verify(p[:1], q[:1], d[:1], t[:1], w.seed, nthreads=1)
    dt1 = time.perf_counter() - t1
    base = {"value": w.B * w.K * w.gamma / dt, "unit": UNIT, "cores": nt, "kind": "oracle",
            "single_thread": w.K * w.gamma / dt1, "cpu": "%s, %d cores" % (cpu_model(), cores),
            "sample": "all %d sequences of the same workload, one thread per sequence "
                      "(%.1f s wall); single_thread: the first sequence on one thread "
                      "(%.1f s)" % (w.B, dt, dt1)}
    return base, (parity_block(gpu, orc) if gpu is not None else None)


# ---------------------------------------------------------------------------
# the reference arm: the fp64 CPU oracle as it stands
# ---------------------------------------------------------------------------

def run_reference(args):
    import oracle
    oracle.lib()
    pool = 4
    c = synth.CONFIGS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    # the first `pool` sequences of the same workload (same generator and seed)
    w = synth.workload(args.workload, device=dev, seed=args.workload, B=min(pool, c["B"]))
    p, q, d, t = synth.to_oracle_arrays(w)
    del w
    if dev == "cuda":
        torch.cuda.empty_cache()
    nt = oracle.max_threads()
    tokens = c["K"] * c["gamma"]

    def step(i):
        b = i % p.shape[0]
        oracle.verify(p[b:b + 1], q[b:b + 1], d[b:b + 1], t[b:b + 1], 0, b0=b, nthreads=nt)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = tokens * args.steps / dt
    sample = ("one sequence (%d x %d rows of V = %d) per step, cycling over the first %d sequences "
              "of the workload; rows spread over %d threads" % (c["K"], 2 * c["gamma"] + 1, c["V"],
                                                                 p.shape[0], nt))
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded logits and drafts; no model weights)",
        "config": {"workload": c["name"], "B": c["B"], "K": c["K"], "gamma": c["gamma"], "V": c["V"],
                   "parallelism": "host cores (fp64 CPU oracle)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    rank, world, local = dist_setup()
    if args.decode_step:
        res = run_decode_step(args, rank, world)
    elif args.cps:
        res = run_cps(args, rank, world)
    else:
        res = run_sdv(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
