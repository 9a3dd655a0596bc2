"""fp64 CPU oracle of batched lossless draft verification with self-selection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library; the C source ``sdv_oracle.c`` states which passages of
"SpecDiff-2: Scaling Diffusion Drafter Alignment For Faster Speculative
Decoding" and "DiffuSpec: Unlocking Diffusion Language Models for Speculative
Decoding" each function follows.

All arrays are numpy; logits are given as raw bf16 words (``uint16``) or
``float32``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

BF16, F32 = 0, 1
BAND_ACCEPT, BAND_CDF, BAND_SELECT, BAND_RESID = 1, 2, 4, 8
BAD_DRAFT, BAD_ROW, BAD_TEMP = 1, 2, 4

_lib = None


def lib():
    """Load (building on first use) the oracle shared library."""
    global _lib
    if _lib is None:
        # SDV_ORACLE_LIB lets the mutation test load a deliberately broken copy.
        path = os.environ.get("SDV_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        dp = ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        L.sdvo_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.sdvo_philox4x32_10.restype = None
        L.sdvo_uniform24.argtypes = [ctypes.c_uint32]
        L.sdvo_uniform24.restype = ctypes.c_double
        L.sdvo_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, dp, dp]
        L.sdvo_uniforms.restype = None
        L.sdvo_row_lse.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.c_double]
        L.sdvo_row_lse.restype = ctypes.c_double
        L.sdvo_accept_ratio.argtypes = [ctypes.c_double, ctypes.c_double]
        L.sdvo_accept_ratio.restype = ctypes.c_double
        L.sdvo_streak_score.argtypes = [dp, ctypes.c_int]
        L.sdvo_streak_score.restype = ctypes.c_double
        L.sdvo_argmax_first.argtypes = [dp, ctypes.c_int]
        L.sdvo_argmax_first.restype = ctypes.c_int
        L.sdvo_accept_length.argtypes = [dp, dp, ctypes.c_int]
        L.sdvo_accept_length.restype = ctypes.c_int
        L.sdvo_inverse_cdf.argtypes = [dp, ctypes.c_int64, ctypes.c_double, dp, dp, dp, dp]
        L.sdvo_inverse_cdf.restype = ctypes.c_int64
        common = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                  vp, vp, vp, vp]
        outs = [vp] * 9 + [ctypes.c_int]
        L.sdvo_verify_uniforms.argtypes = common + [vp, vp] + outs
        L.sdvo_verify_uniforms.restype = ctypes.c_int
        L.sdvo_verify.argtypes = common + [ctypes.c_uint64, ctypes.c_int32] + outs
        L.sdvo_verify.restype = ctypes.c_int
        L.sdvo_verify_greedy_uniforms.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int64, ctypes.c_int, vp, vp, vp, vp,
                                                  vp] + outs
        L.sdvo_verify_greedy_uniforms.restype = ctypes.c_int
        L.sdvo_verify_greedy.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                         ctypes.c_int, vp, vp, vp, ctypes.c_uint64,
                                         ctypes.c_int32] + outs
        L.sdvo_verify_greedy.restype = ctypes.c_int
        L.sdvo_verify_lens.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                       ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp,
                                       ctypes.c_uint64, ctypes.c_int32] + outs
        L.sdvo_verify_lens.restype = ctypes.c_int
        L.sdvo_accept_ratio_greedy.argtypes = [ctypes.c_double]
        L.sdvo_accept_ratio_greedy.restype = ctypes.c_double
        L.sdvo_cps_prune_row.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                                         ctypes.c_double, ctypes.c_int, vp, vp, dp, dp]
        L.sdvo_cps_prune_row.restype = ctypes.c_int
        L.sdvo_cps.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int, vp, vp,
                               ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int32,
                               vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
        L.sdvo_cps.restype = ctypes.c_int
        L.sdvo_adl_state_words.argtypes = [ctypes.c_int]
        L.sdvo_adl_state_words.restype = ctypes.c_int
        L.sdvo_adl_step.argtypes = [ctypes.c_int] * 6 + [vp, vp, vp, vp]
        L.sdvo_adl_step.restype = ctypes.c_int
        L.sdvo_max_threads.argtypes = []
        L.sdvo_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def philox4x32_10(ctr, key):
    """Philox4x32-10 block function: 4 counter words, 2 key words -> 4 words."""
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xffffffff for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xffffffff for x in key])
    o = (ctypes.c_uint32 * 4)()
    lib().sdvo_philox4x32_10(c, k, o)
    return [int(x) for x in o]


def uniform24(word):
    return lib().sdvo_uniform24(int(word) & 0xffffffff)


def uniforms(seed, b, j):
    """(u, w) for sequence b, position j under the (j, b, 0, 0) counter keying."""
    u, w = ctypes.c_double(), ctypes.c_double()
    lib().sdvo_uniforms(int(seed), int(b), int(j), ctypes.byref(u), ctypes.byref(w))
    return u.value, w.value


def _row_dtype(row):
    row = np.ascontiguousarray(row)
    if row.dtype == np.uint16:
        return row, BF16
    if row.dtype == np.float32:
        return row, F32
    raise TypeError("rows are raw bf16 words (uint16) or float32")


def row_lse(row, T=1.0):
    row, dt = _row_dtype(row)
    return lib().sdvo_row_lse(_ptr(row), dt, row.shape[-1], float(T))


def accept_ratio(lp, lq):
    return lib().sdvo_accept_ratio(float(lp), float(lq))


def streak_score(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return lib().sdvo_streak_score(a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), a.shape[0])


def argmax_first(s):
    s = np.ascontiguousarray(s, dtype=np.float64)
    return lib().sdvo_argmax_first(s.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), s.shape[0])


def accept_length(a, u):
    a = np.ascontiguousarray(a, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    return lib().sdvo_accept_length(a.ctypes.data_as(dp), u.ctypes.data_as(dp), a.shape[0])


def inverse_cdf(r, w):
    """Returns (v, R, t, C_{v-1}, C_v)."""
    r = np.ascontiguousarray(r, dtype=np.float64)
    R, t, cp, cv = (ctypes.c_double() for _ in range(4))
    v = lib().sdvo_inverse_cdf(r.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), r.shape[0],
                               float(w), ctypes.byref(R), ctypes.byref(t), ctypes.byref(cp),
                               ctypes.byref(cv))
    return int(v), R.value, t.value, cp.value, cv.value


def _verify_common(p_logits, q_logits, drafts, temps):
    p_logits = np.ascontiguousarray(p_logits)
    q_logits = np.ascontiguousarray(q_logits)
    if p_logits.dtype != q_logits.dtype:
        raise TypeError("p and q logits must share a dtype")
    _, dt = _row_dtype(p_logits[..., :1].reshape(-1)[:1])
    B, K, G1, V = p_logits.shape
    G = G1 - 1
    if q_logits.shape != (B, K, G, V):
        raise ValueError("q_logits must be [B, K, gamma, V]")
    drafts = np.ascontiguousarray(drafts, dtype=np.int32)
    if drafts.shape != (B, K, G):
        raise ValueError("drafts must be [B, K, gamma]")
    temps = np.broadcast_to(np.asarray(temps, dtype=np.float64), (B,)).copy()
    out = dict(
        sel=np.full(B, -1, np.int32), accept_len=np.full(B, -1, np.int32),
        next_token=np.full(B, -1, np.int32), lse=np.zeros((B, K, 2 * G + 1)),
        scores=np.zeros((B, K)), ratio=np.zeros((B, K, max(G, 1))),
        band=np.zeros(B, np.int32), err=np.zeros(B, np.int32), resid_mass=np.zeros(B))
    return p_logits, q_logits, drafts, temps, dt, (B, K, G, V), out


_OUT_ORDER = ("sel", "accept_len", "next_token", "lse", "scores", "ratio", "band", "err",
              "resid_mass")


def _outs(out, nthreads):
    return [_ptr(out[k]) for k in _OUT_ORDER] + [int(nthreads)]


def _lens(lens, B):
    return None if lens is None else np.ascontiguousarray(
        np.broadcast_to(np.asarray(lens, dtype=np.int32), (B,)))


def verify(p_logits, q_logits, drafts, temps, seed, b0=0, nthreads=1, lens=None):
    """Full step with Philox uniforms keyed by (seed, b0 + b, j).

    p_logits [B,K,gamma+1,V] and q_logits [B,K,gamma,V] as uint16 (bf16 words)
    or float32; drafts [B,K,gamma] int; temps scalar or [B]; lens None or the
    draft length of each sequence [B] (0..gamma; positions past it are not
    read).  Returns a dict of numpy arrays: sel, accept_len, next_token, lse,
    scores, ratio, band, err, resid_mass.
    """
    p, q, d, t, dt, (B, K, G, V), out = _verify_common(p_logits, q_logits, drafts, temps)
    if lens is None:
        lib().sdvo_verify(B, K, G, V, dt, _ptr(p), _ptr(q), _ptr(d), _ptr(t), int(seed),
                          int(b0), *_outs(out, nthreads))
    else:
        ln = _lens(lens, B)
        lib().sdvo_verify_lens(B, K, G, V, dt, 0, _ptr(p), _ptr(q), _ptr(d), _ptr(t), _ptr(ln),
                               int(seed), int(b0), *_outs(out, nthreads))
    if G == 0:
        out["ratio"] = out["ratio"][..., :0]
    return out


def verify_uniforms(p_logits, q_logits, drafts, temps, u, w, nthreads=1):
    """Full step with explicit uniforms u [B,gamma] and w [B,gamma+1]."""
    p, q, d, t, dt, (B, K, G, V), out = _verify_common(p_logits, q_logits, drafts, temps)
    u = np.ascontiguousarray(np.broadcast_to(np.asarray(u, np.float64), (B, G)))
    w = np.ascontiguousarray(np.broadcast_to(np.asarray(w, np.float64), (B, G + 1)))
    lib().sdvo_verify_uniforms(B, K, G, V, dt, _ptr(p), _ptr(q), _ptr(d), _ptr(t), _ptr(u),
                               _ptr(w), *_outs(out, nthreads))
    if G == 0:
        out["ratio"] = out["ratio"][..., :0]
    return out


def _greedy_common(p_logits, drafts, temps):
    p_logits = np.ascontiguousarray(p_logits)
    _, dt = _row_dtype(p_logits[..., :1].reshape(-1)[:1])
    B, K, G1, V = p_logits.shape
    G = G1 - 1
    drafts = np.ascontiguousarray(drafts, dtype=np.int32)
    if drafts.shape != (B, K, G):
        raise ValueError("drafts must be [B, K, gamma]")
    temps = np.broadcast_to(np.asarray(temps, dtype=np.float64), (B,)).copy()
    out = dict(
        sel=np.full(B, -1, np.int32), accept_len=np.full(B, -1, np.int32),
        next_token=np.full(B, -1, np.int32), lse=np.zeros((B, K, 2 * G + 1)),
        scores=np.zeros((B, K)), ratio=np.zeros((B, K, max(G, 1))),
        band=np.zeros(B, np.int32), err=np.zeros(B, np.int32), resid_mass=np.zeros(B))
    return p_logits, drafts, temps, dt, (B, K, G, V), out


def verify_greedy(p_logits, drafts, temps, seed, b0=0, nthreads=1, lens=None):
    """Greedy acceptance (no drafter rows), Philox uniforms and lens as verify()."""
    p, d, t, dt, (B, K, G, V), out = _greedy_common(p_logits, drafts, temps)
    if lens is None:
        lib().sdvo_verify_greedy(B, K, G, V, dt, _ptr(p), _ptr(d), _ptr(t), int(seed), int(b0),
                                 *_outs(out, nthreads))
    else:
        ln = _lens(lens, B)
        lib().sdvo_verify_lens(B, K, G, V, dt, 1, _ptr(p), None, _ptr(d), _ptr(t), _ptr(ln),
                               int(seed), int(b0), *_outs(out, nthreads))
    return out


def verify_greedy_uniforms(p_logits, drafts, temps, u, w, nthreads=1):
    """Greedy acceptance with explicit uniforms u [B,gamma], w [B,gamma+1]."""
    p, d, t, dt, (B, K, G, V), out = _greedy_common(p_logits, drafts, temps)
    u = np.ascontiguousarray(np.broadcast_to(np.asarray(u, np.float64), (B, G)))
    w = np.ascontiguousarray(np.broadcast_to(np.asarray(w, np.float64), (B, G + 1)))
    lib().sdvo_verify_greedy_uniforms(B, K, G, V, dt, _ptr(p), _ptr(d), _ptr(t), _ptr(u),
                                      _ptr(w), *_outs(out, nthreads))
    return out


def accept_ratio_greedy(lp):
    return lib().sdvo_accept_ratio_greedy(float(lp))


CPS_BAND_MASS = 1


def cps_prune_row(row, T, tau, mmax):
    """Candidates of one drafter row: (ids, natural-log probs, mass without
    the last kept token, mass with it)."""
    row, dt = _row_dtype(row)
    ids = np.full(mmax, -1, np.int32)
    lp = np.full(mmax, -np.inf)
    mb, ma = ctypes.c_double(), ctypes.c_double()
    n = lib().sdvo_cps_prune_row(_ptr(row), dt, row.shape[-1], float(T), float(tau), int(mmax),
                                 _ptr(ids), _ptr(lp), ctypes.byref(mb), ctypes.byref(ma))
    return ids[:n], lp[:n], mb.value, ma.value


def cps(q, temps, tau, mmax, beam, eos_id=-1, nthreads=1):
    """Causal-consistency path search over drafter marginals q [B, gamma, V]
    (uint16 bf16 words or float32).  Returns a dict: cand_ids, cand_logp,
    ncand, lat_len, paths, path_logp, npaths, band."""
    q = np.ascontiguousarray(q)
    _, dt = _row_dtype(q[..., :1].reshape(-1)[:1])
    B, G, V = q.shape
    temps = np.broadcast_to(np.asarray(temps, dtype=np.float64), (B,)).copy()
    out = dict(cand_ids=np.full((B, G, mmax), -1, np.int32), cand_logp=np.zeros((B, G, mmax)),
               ncand=np.zeros((B, G), np.int32), lat_len=np.zeros(B, np.int32),
               paths=np.full((B, beam, G), -1, np.int32), path_logp=np.zeros((B, beam)),
               npaths=np.zeros(B, np.int32), band=np.zeros(B, np.int32))
    st = lib().sdvo_cps(B, G, V, dt, _ptr(q), _ptr(temps), float(tau), int(mmax), int(beam),
                        int(eos_id), _ptr(out["cand_ids"]), _ptr(out["cand_logp"]),
                        _ptr(out["ncand"]), _ptr(out["lat_len"]), _ptr(out["paths"]),
                        _ptr(out["path_logp"]), _ptr(out["npaths"]), _ptr(out["band"]),
                        int(nthreads))
    if st != 0:
        raise RuntimeError("oracle cps failed")
    return out


def adl_state(B, W):
    """Zeroed controller state for B sequences and window W."""
    return np.zeros((B, lib().sdvo_adl_state_words(int(W))), np.int32)


def adl_step(k, gen_len, acc_len, state, W=1, kmin=1, kmax=64, up=2, down=1):
    """One adaptive-draft-length step: returns the next draft lengths [B] and
    updates `state` (from adl_state) in place."""
    k = np.ascontiguousarray(k, dtype=np.int32).copy()
    g = np.ascontiguousarray(gen_len, dtype=np.int32)
    a = np.ascontiguousarray(acc_len, dtype=np.int32)
    assert state.dtype == np.int32 and state.flags.c_contiguous
    st = lib().sdvo_adl_step(len(k), int(W), int(kmin), int(kmax), int(up), int(down), _ptr(g),
                             _ptr(a), _ptr(k), _ptr(state))
    if st != 0:
        raise ValueError("oracle adl_step: invalid parameters")
    return k


def max_threads():
    return lib().sdvo_max_threads()
