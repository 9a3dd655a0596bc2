"""ctypes binding of libsdv (``include/sdv.h``), torch tensors in and out.

Argument marshalling only: every step of the verification runs in the CUDA
kernels of ``libsdv.so``.  There is no fallback: if the library is missing or
does not load, every call raises.

The functions keep the C names (``sdv_create``, ``sdv_verify``,
``sdv_verify_ex``, ``sdv_verify_host``, ``sdv_sync``, ``sdv_last_error``,
``sdv_destroy``, ``sdv_plan``); ``Verifier`` wraps a context.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsdv.so")

SDV_OK, SDV_ERR_ARG, SDV_ERR_CUDA, SDV_ERR_OOM, SDV_ERR_DEVICE_DATA, SDV_ERR_SCRATCH = 0, 1, 2, 3, 4, 5
SDV_BF16, SDV_F32 = 0, 1
SDV_FLAG_SHARED_Q = 1
SDV_FLAG_GREEDY = 2
SDV_FLAG_SHARED_PREFIX_ROW = 4
STATUS_NAMES = {0: "SDV_OK", 1: "SDV_ERR_ARG", 2: "SDV_ERR_CUDA", 3: "SDV_ERR_OOM",
                4: "SDV_ERR_DEVICE_DATA", 5: "SDV_ERR_SCRATCH"}
STATIC_SCRATCH_BYTES = 8 << 20
SDV_STATUS_BAD_LENGTH = 16
SDV_HOOK_SAMPLE_NO_COPY = 1

# Every entry point of include/sdv.h, with its ctypes signature.
_VP, _I, _I64, _U64, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
SIGNATURES = {
    "sdv_create": (_I, [ctypes.POINTER(_VP), _I, _I, _I, _I, _I, _VP]),
    "sdv_create_ex": (_I, [ctypes.POINTER(_VP), _I, _I, _I, _I, _I, _VP, ctypes.c_uint]),
    "sdv_verify": (_I, [_VP, _VP, _VP, _VP, _F, _U64, _VP, _VP, _VP]),
    "sdv_verify_ex": (_I, [_VP, _VP, _VP, _VP, _F, _VP, _U64, _VP, _VP, _VP, _VP, _VP]),
    "sdv_verify_len": (_I, [_VP, _VP, _VP, _VP, _VP, _F, _VP, _U64, _VP, _VP, _VP, _VP, _VP]),
    "sdv_verify_qstat": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _F, _VP, _U64, _VP, _VP, _VP, _VP,
                              _VP]),
    "sdv_verify_host": (_I, [_VP, _VP, _VP, _VP, _F, _VP, _U64, _VP, _VP, _VP]),
    "sdv_sync": (_I, [_VP]),
    "sdv_last_error": (ctypes.c_char_p, [_VP]),
    "sdv_destroy": (None, [_VP]),
    "sdv_plan": (_I, [_VP, ctypes.POINTER(_I), ctypes.POINTER(_I64), ctypes.POINTER(_I),
                      ctypes.POINTER(_I)]),
    "sdv_set_stream": (_I, [_VP, _VP]),
    "sdv_set_test_hooks": (_I, [_VP, ctypes.c_uint]),
    "sdv_profile_enable": (_I, [_VP, _I]),
    "sdv_profile_read": (_I, [_VP, ctypes.POINTER(_F), ctypes.POINTER(_I)]),
    "sdv_verify_static": (_I, [_I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _F, _VP, _U64, _VP, _VP, _VP]),
    "sdv_cps": (_I, [_I, _I, _I, _I, _VP, _VP, _F, _VP, _F, _I, _I, _I, _VP, _VP, _VP, _VP, _VP,
                     _VP, _VP, _VP]),
    "sdv_cps_ex": (_I, [_I, _I, _I, _I, _VP, _VP, _F, _VP, _F, _I, _I, _I, _VP, _VP, _VP, _VP,
                        _VP, _VP, _VP, _VP, _VP]),
    "sdv_cps_prune": (_I, [_I, _I, _I, _I, _VP, _VP, _F, _VP, _F, _I, _VP, _VP, _VP, _VP]),
    "sdv_cps_beam": (_I, [_I, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "sdv_adl_state_words": (_I, [_I]),
    "sdv_adl_step_host": (_I, [_I, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP]),
    "sdv_adl_step": (_I, [_I, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP]),
}

_lib = None


class SdvError(RuntimeError):
    def __init__(self, status: int, msg: str = ""):
        super().__init__("%s%s" % (STATUS_NAMES.get(status, str(status)), (": " + msg) if msg else ""))
        self.status = status


def load(build: bool = False) -> ctypes.CDLL:
    """Load libsdv.so (optionally building it first).  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if build:
        from . import build as _b
        _b.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libsdv.so is not built (run draft_verification_sdv_gb300.build.build());"
                           " there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _dev_ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def _per_seq(t: Optional[torch.Tensor], B: int, name: str) -> None:
    """A per-sequence array must hold one entry per sequence: the library
    reads B of them."""
    if t is not None and t.numel() != B:
        raise ValueError("%s must have one entry per sequence (%d)" % (name, B))


def _host_ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("%s must be a host tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return SDV_BF16
    if dtype == torch.float32:
        return SDV_F32
    raise TypeError("logits must be bfloat16 or float32")


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def sdv_create(B: int, K: int, gamma: int, V: int, dtype: torch.dtype = torch.bfloat16,
               stream=None, flags: int = 0) -> ctypes.c_void_p:
    ctx = ctypes.c_void_p()
    st = load().sdv_create_ex(ctypes.byref(ctx), B, K, gamma, V, _dtype_code(dtype),
                              ctypes.c_void_p(_stream_handle(stream)), int(flags))
    if st != SDV_OK:
        raise SdvError(st, "sdv_create(B=%d, K=%d, gamma=%d, V=%d)" % (B, K, gamma, V))
    return ctx


def sdv_verify(ctx, p_logits, q_logits, drafts, temperature, seed, out_sel, out_accept_len,
               out_next_token) -> int:
    return load().sdv_verify(ctx, _dev_ptr(p_logits, name="p_logits"),
                             _dev_ptr(q_logits, name="q_logits"),
                             _dev_ptr(drafts, torch.int32, "drafts"), float(temperature),
                             int(seed) & 0xFFFFFFFFFFFFFFFF, _dev_ptr(out_sel, torch.int32, "out_sel"),
                             _dev_ptr(out_accept_len, torch.int32, "out_accept_len"),
                             _dev_ptr(out_next_token, torch.int32, "out_next_token"))


def sdv_verify_ex(ctx, p_logits, q_logits, drafts, temperature, temperature_per_seq, seed,
                  out_sel, out_accept_len, out_next_token, out_scores=None, out_lse=None) -> int:
    return load().sdv_verify_ex(
        ctx, _dev_ptr(p_logits, name="p_logits"), _dev_ptr(q_logits, name="q_logits"),
        _dev_ptr(drafts, torch.int32, "drafts"), float(temperature),
        _dev_ptr(temperature_per_seq, torch.float32, "temperature_per_seq"),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev_ptr(out_sel, torch.int32, "out_sel"),
        _dev_ptr(out_accept_len, torch.int32, "out_accept_len"),
        _dev_ptr(out_next_token, torch.int32, "out_next_token"),
        _dev_ptr(out_scores, torch.float32, "out_scores"),
        _dev_ptr(out_lse, torch.float32, "out_lse"))


def sdv_verify_qstat(ctx, p_logits, q_logits, drafts, draft_len, q_row_stat, temperature,
                     temperature_per_seq, seed, out_sel, out_accept_len, out_next_token,
                     out_scores=None, out_lse=None) -> int:
    return load().sdv_verify_qstat(
        ctx, _dev_ptr(p_logits, name="p_logits"), _dev_ptr(q_logits, name="q_logits"),
        _dev_ptr(drafts, torch.int32, "drafts"), _dev_ptr(draft_len, torch.int32, "draft_len"),
        _dev_ptr(q_row_stat, torch.float32, "q_row_stat"), float(temperature),
        _dev_ptr(temperature_per_seq, torch.float32, "temperature_per_seq"),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev_ptr(out_sel, torch.int32, "out_sel"),
        _dev_ptr(out_accept_len, torch.int32, "out_accept_len"),
        _dev_ptr(out_next_token, torch.int32, "out_next_token"),
        _dev_ptr(out_scores, torch.float32, "out_scores"),
        _dev_ptr(out_lse, torch.float32, "out_lse"))


def sdv_verify_len(ctx, p_logits, q_logits, drafts, draft_len, temperature, temperature_per_seq,
                   seed, out_sel, out_accept_len, out_next_token, out_scores=None,
                   out_lse=None) -> int:
    return load().sdv_verify_len(
        ctx, _dev_ptr(p_logits, name="p_logits"), _dev_ptr(q_logits, name="q_logits"),
        _dev_ptr(drafts, torch.int32, "drafts"), _dev_ptr(draft_len, torch.int32, "draft_len"),
        float(temperature), _dev_ptr(temperature_per_seq, torch.float32, "temperature_per_seq"),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev_ptr(out_sel, torch.int32, "out_sel"),
        _dev_ptr(out_accept_len, torch.int32, "out_accept_len"),
        _dev_ptr(out_next_token, torch.int32, "out_next_token"),
        _dev_ptr(out_scores, torch.float32, "out_scores"),
        _dev_ptr(out_lse, torch.float32, "out_lse"))


def sdv_verify_host(ctx, p_logits, q_logits, drafts, temperature, temperature_per_seq, seed,
                    out_sel, out_accept_len, out_next_token) -> int:
    return load().sdv_verify_host(
        ctx, _host_ptr(p_logits, name="p_logits"), _host_ptr(q_logits, name="q_logits"),
        _host_ptr(drafts, torch.int32, "drafts"), float(temperature),
        _host_ptr(temperature_per_seq, torch.float32, "temperature_per_seq"),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _host_ptr(out_sel, torch.int32, "out_sel"),
        _host_ptr(out_accept_len, torch.int32, "out_accept_len"),
        _host_ptr(out_next_token, torch.int32, "out_next_token"))


def sdv_sync(ctx) -> int:
    return load().sdv_sync(ctx)


def sdv_last_error(ctx) -> str:
    r = load().sdv_last_error(ctx)
    return r.decode() if r else ""


def sdv_destroy(ctx) -> None:
    load().sdv_destroy(ctx)


def sdv_plan(ctx) -> dict:
    g, ck, cv, cl = _I(), _I(), _I64(), _I()
    st = load().sdv_plan(ctx, ctypes.byref(g), ctypes.byref(cv), ctypes.byref(ck), ctypes.byref(cl))
    if st != SDV_OK:
        raise SdvError(st)
    return {"rowpass_ctas": g.value, "chunk_vectors": cv.value, "chunks_per_row": ck.value,
            "sample_cluster": cl.value}


def sdv_profile_enable(ctx, enable: bool = True) -> int:
    return load().sdv_profile_enable(ctx, 1 if enable else 0)


def sdv_profile_read(ctx):
    """(mean ms of [row pass, select, sample], number of steps); clears the record."""
    ms = (_F * 3)()
    n = _I()
    st = load().sdv_profile_read(ctx, ms, ctypes.byref(n))
    if st != SDV_OK:
        raise SdvError(st, sdv_last_error(ctx))
    return [float(x) for x in ms], n.value


def sdv_verify_static(B, K, gamma, V, dtype, stream, p_logits, q_logits, drafts, temperature,
                      temperature_per_seq, seed, out_sel, out_accept_len, out_next_token) -> int:
    """Allocation-free step (no context): scratch lives in a static device array."""
    return load().sdv_verify_static(
        B, K, gamma, V, _dtype_code(dtype), ctypes.c_void_p(_stream_handle(stream)),
        _dev_ptr(p_logits, name="p_logits"), _dev_ptr(q_logits, name="q_logits"),
        _dev_ptr(drafts, torch.int32, "drafts"), float(temperature),
        _dev_ptr(temperature_per_seq, torch.float32, "temperature_per_seq"),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _dev_ptr(out_sel, torch.int32, "out_sel"),
        _dev_ptr(out_accept_len, torch.int32, "out_accept_len"),
        _dev_ptr(out_next_token, torch.int32, "out_next_token"))


def sdv_cps(q_marginals, tau: float = 0.8, mmax: int = 15, beam: int = 3, eos_id: int = -1,
            temperature: float = 1.0, temps: Optional[torch.Tensor] = None, stream=None,
            out: Optional[dict] = None, row_stat: bool = False) -> dict:
    """Causal-consistency path search over drafter marginals q [B, gamma, V]
    (candidate pruning by cumulative mass, EOS cut, beam by drafter
    confidence).  Enqueues on `stream` (default: the current stream) and
    returns the output tensors; `out` (a dict this returned for the same
    shapes) reuses them.  With `row_stat`, out["row_stat"] [B, gamma, 4] holds
    each marginal row's softmax statistics (sdv_cps_ex), which a Verifier call
    takes as `q_stat` so that it does not stream the marginals again."""
    B, G, V = q_marginals.shape
    _per_seq(temps, B, "temps")
    dev = q_marginals.device
    if out is not None and row_stat and "row_stat" not in out:
        out["row_stat"] = torch.empty((B, G, 4), dtype=torch.float32, device=dev)
    out = out if out is not None else {
        "cand_ids": torch.empty((B, G, mmax), dtype=torch.int32, device=dev),
        "cand_logp": torch.empty((B, G, mmax), dtype=torch.float32, device=dev),
        "cand_logit": torch.empty((B, G, mmax), dtype=torch.float32, device=dev),
        "ncand": torch.empty((B, G), dtype=torch.int32, device=dev),
        "paths": torch.empty((B, beam, G), dtype=torch.int32, device=dev),
        "path_logp": torch.empty((B, beam), dtype=torch.float32, device=dev),
        "npaths": torch.empty((B,), dtype=torch.int32, device=dev),
        "lat_len": torch.empty((B,), dtype=torch.int32, device=dev),
    }
    if row_stat and "row_stat" not in out:
        out["row_stat"] = torch.empty((B, G, 4), dtype=torch.float32, device=dev)
    st = load().sdv_cps_ex(B, G, V, _dtype_code(q_marginals.dtype),
                           ctypes.c_void_p(_stream_handle(stream)),
                           _dev_ptr(q_marginals, name="q_marginals"), float(temperature),
                           _dev_ptr(temps, torch.float32, "temps"), float(tau), int(mmax), int(beam),
                           int(eos_id), *[_dev_ptr(out[k]) for k in ("cand_ids", "cand_logp",
                                                                     "cand_logit", "ncand", "paths",
                                                                     "path_logp", "npaths",
                                                                     "lat_len")],
                           _dev_ptr(out["row_stat"], torch.float32, "row_stat") if row_stat else None)
    if st != SDV_OK:
        raise SdvError(st, "sdv_cps")
    return out


def _cps_lattice(B, G, mmax, dev):
    return {"cand_ids": torch.empty((B, G, mmax), dtype=torch.int32, device=dev),
            "cand_logp": torch.empty((B, G, mmax), dtype=torch.float32, device=dev),
            "cand_logit": torch.empty((B, G, mmax), dtype=torch.float32, device=dev),
            "ncand": torch.empty((B, G), dtype=torch.int32, device=dev)}


def sdv_cps_prune(q_marginals, tau: float = 0.8, mmax: int = 15, temperature: float = 1.0,
                  temps: Optional[torch.Tensor] = None, stream=None, out: Optional[dict] = None) -> dict:
    """The pruning half of sdv_cps: every row's candidate list (no EOS cut).
    `out` (the dict this returns) may be passed back to reuse its tensors."""
    B, G, V = q_marginals.shape
    _per_seq(temps, B, "temps")
    out = out if out is not None else _cps_lattice(B, G, mmax, q_marginals.device)
    st = load().sdv_cps_prune(B, G, V, _dtype_code(q_marginals.dtype),
                              ctypes.c_void_p(_stream_handle(stream)),
                              _dev_ptr(q_marginals, name="q_marginals"), float(temperature),
                              _dev_ptr(temps, torch.float32, "temps"), float(tau), int(mmax),
                              *[_dev_ptr(out[k]) for k in ("cand_ids", "cand_logp", "cand_logit",
                                                           "ncand")])
    if st != SDV_OK:
        raise SdvError(st, "sdv_cps_prune")
    return out


def sdv_cps_beam(lattice: dict, V: int, beam: int = 3, eos_id: int = -1, stream=None,
                 out: Optional[dict] = None) -> dict:
    """The beam half of sdv_cps over a lattice from sdv_cps_prune (trimmed in
    place at an EOS end).  Returns the lattice dict with the path tensors;
    `out` (a dict this returned for the same shapes) reuses them."""
    B, G, mmax = lattice["cand_ids"].shape
    dev = lattice["cand_ids"].device
    if out is None:
        out = dict(lattice)
        out.update({"paths": torch.empty((B, beam, G), dtype=torch.int32, device=dev),
                    "path_logp": torch.empty((B, beam), dtype=torch.float32, device=dev),
                    "npaths": torch.empty((B,), dtype=torch.int32, device=dev),
                    "lat_len": torch.empty((B,), dtype=torch.int32, device=dev)})
    else:
        out.update(lattice)
    st = load().sdv_cps_beam(B, G, int(V), int(mmax), int(beam), int(eos_id),
                             ctypes.c_void_p(_stream_handle(stream)),
                             *[_dev_ptr(out[k]) for k in ("cand_ids", "cand_logp", "cand_logit",
                                                          "ncand", "paths",
                                                          "path_logp", "npaths", "lat_len")])
    if st != SDV_OK:
        raise SdvError(st, "sdv_cps_beam")
    return out


class DraftLengthController:
    """Adaptive draft length for B sequences (the library's rule; see
    sdv_adl_step in include/sdv.h).  On a CUDA device the state, the lengths
    and the update stay on the device (`step` enqueues one kernel); on the
    host the same rule runs in the library's C code."""

    def __init__(self, B: int, k0, window: int = 1, kmin: int = 1, kmax: int = 64, up: int = 2,
                 down: int = 1, device="cuda"):
        words = load().sdv_adl_state_words(int(window))
        if words < 0:
            raise SdvError(SDV_ERR_ARG, "window")
        self.B, self.window, self.kmin, self.kmax, self.up, self.down = B, window, kmin, kmax, up, down
        self.device = torch.device(device)
        self.state = torch.zeros((B, words), dtype=torch.int32, device=self.device)
        self.k = torch.as_tensor(k0, dtype=torch.int32).expand(B).clone().to(self.device)
        self.status = (torch.zeros(1, dtype=torch.int32, device=self.device)
                       if self.device.type == "cuda" else None)

    def step(self, gen_len: torch.Tensor, acc_len: torch.Tensor, stream=None) -> torch.Tensor:
        """Record one step's generated and accepted lengths [B] (int32, on the
        controller's device) and return the next draft lengths (self.k)."""
        _per_seq(gen_len, self.B, "gen_len")
        _per_seq(acc_len, self.B, "acc_len")
        g = gen_len.to(torch.int32).contiguous()
        a = acc_len.to(torch.int32).contiguous()
        if self.device.type == "cuda":
            st = load().sdv_adl_step(self.B, self.window, self.kmin, self.kmax, self.up, self.down,
                                     ctypes.c_void_p(_stream_handle(stream)), _dev_ptr(g), _dev_ptr(a),
                                     _dev_ptr(self.k), _dev_ptr(self.state), _dev_ptr(self.status))
        else:
            st = load().sdv_adl_step_host(self.B, self.window, self.kmin, self.kmax, self.up,
                                          self.down, _host_ptr(g), _host_ptr(a), _host_ptr(self.k),
                                          _host_ptr(self.state))
        if st != SDV_OK:
            raise SdvError(st, "sdv_adl_step")
        return self.k


def sdv_set_stream(ctx, stream) -> int:
    return load().sdv_set_stream(ctx, ctypes.c_void_p(_stream_handle(stream)))


def sdv_set_test_hooks(ctx, hooks: int) -> int:
    """Fault-path test hooks of a context (SDV_HOOK_* bits; 0 = none)."""
    return load().sdv_set_test_hooks(ctx, int(hooks))


class Verifier:
    """One context for batches of shape (B, K, gamma, V).

    ``v(p, q, drafts, ...)`` enqueues a step on the context's stream and returns
    the output tensors; ``v.sync()`` waits and raises on a device-side error.
    """

    def __init__(self, B: int, K: int, gamma: int, V: int, dtype=torch.bfloat16,
                 device=None, stream=None, shared_q: bool = False, greedy: bool = False,
                 shared_prefix_row: bool = False):
        self.B, self.K, self.gamma, self.V, self.dtype = B, K, gamma, V, dtype
        self.shared_q = shared_q
        self.greedy = greedy
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        with torch.cuda.device(self.device):
            self.stream = stream
            self.ctx = sdv_create(B, K, gamma, V, dtype, stream,
                                  (SDV_FLAG_SHARED_Q if shared_q else 0) |
                                  (SDV_FLAG_GREEDY if greedy else 0) |
                                  (SDV_FLAG_SHARED_PREFIX_ROW if shared_prefix_row else 0))

    def __call__(self, p_logits, q_logits, drafts, temperature: float = 1.0, seed: int = 0,
                 temps: Optional[torch.Tensor] = None, scores: bool = False, lse: bool = False,
                 out: Optional[dict] = None, draft_len: Optional[torch.Tensor] = None,
                 q_stat: Optional[torch.Tensor] = None) -> dict:
        """One verification step; `draft_len` (int32 [B] on the device) gives
        each sequence's draft length (sdv_verify_len), else all are gamma;
        `q_stat` (float32 [rows_q, 4], e.g. sdv_cps(..., row_stat=True)
        ["row_stat"]) supplies the drafter rows' softmax statistics, so the
        q rows are not streamed (sdv_verify_qstat)."""
        B, K, G, V = self.B, self.K, self.gamma, self.V
        q_shape = (B, G, V) if self.shared_q else (B, K, G, V)
        if tuple(p_logits.shape) != (B, K, G + 1, V):
            raise ValueError("p_logits must be [B,K,gamma+1,V]")
        if not self.greedy and (q_logits is None or tuple(q_logits.shape) != q_shape):
            raise ValueError("q_logits must be %s" % (list(q_shape),))
        if tuple(drafts.shape) != (B, K, G):
            raise ValueError("drafts must be [B,K,gamma]")
        if p_logits.dtype != self.dtype or (q_logits is not None and q_logits.dtype != self.dtype):
            raise TypeError("logits must be %s" % self.dtype)
        _per_seq(temps, B, "temps")
        _per_seq(draft_len, B, "draft_len")
        dev = p_logits.device
        if out is None:
            out = {
                "sel": torch.empty(B, dtype=torch.int32, device=dev),
                "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
                "next_token": torch.empty(B, dtype=torch.int32, device=dev),
            }
            if scores:
                out["scores"] = torch.empty((B, K), dtype=torch.float32, device=dev)
            if lse:
                out["lse"] = torch.empty((B, K, G + 1 if self.greedy else 2 * G + 1),
                                         dtype=torch.float32, device=dev)
        if q_stat is not None:
            rows_q = B * G if self.shared_q else B * K * G
            if not self.greedy and (q_stat.dtype != torch.float32 or q_stat.numel() != rows_q * 4):
                raise ValueError("q_stat must be float32 with %d x 4 entries (one per q row)"
                                 % rows_q)
            st = sdv_verify_qstat(self.ctx, p_logits, q_logits, drafts, draft_len, q_stat,
                                  temperature, temps, seed, out["sel"], out["accept_len"],
                                  out["next_token"], out.get("scores"), out.get("lse"))
        elif draft_len is None:
            st = sdv_verify_ex(self.ctx, p_logits, q_logits, drafts, temperature, temps, seed,
                               out["sel"], out["accept_len"], out["next_token"], out.get("scores"),
                               out.get("lse"))
        else:
            st = sdv_verify_len(self.ctx, p_logits, q_logits, drafts, draft_len, temperature, temps,
                                seed, out["sel"], out["accept_len"], out["next_token"],
                                out.get("scores"), out.get("lse"))
        if st != SDV_OK:
            raise SdvError(st, sdv_last_error(self.ctx))
        return out

    def set_stream(self, stream) -> None:
        """Enqueue later steps on `stream` (for CUDA-graph capture: the
        capturing stream).  The caller orders it after earlier steps."""
        st = sdv_set_stream(self.ctx, stream)
        if st != SDV_OK:
            raise SdvError(st, sdv_last_error(self.ctx))
        self.stream = stream

    def sync(self) -> None:
        st = sdv_sync(self.ctx)
        if st != SDV_OK:
            raise SdvError(st, sdv_last_error(self.ctx))

    def plan(self) -> dict:
        return sdv_plan(self.ctx)

    def close(self) -> None:
        if getattr(self, "ctx", None) is not None:
            sdv_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
