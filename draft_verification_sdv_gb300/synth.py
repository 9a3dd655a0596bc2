"""Seeded synthetic inputs for batched draft verification.

This module only makes inputs: verifier logits p, drafter logits q and drafts
sampled from softmax(q / T).  It holds none of the verification arithmetic, so
the CUDA path and the CPU oracle can both be fed from it.

The workloads restate the shapes and value distributions of speculative
diffusion decoding with a Qwen2.5 verifier ("SpecDiff-2: Scaling Diffusion
Drafter Alignment For Faster Speculative Decoding", section 6 and appendix
A.3: Qwen2.5 verifiers, windows gamma = 16 / 32, K drafts from one denoising
pass, drafting temperatures around 1).  Synthetic logits stand in for the
models' outputs on the pages' benchmarks:

* verifier row      l_p = N(0, 3^2) + Zipf log-prior -1.1 * ln(v + 1)
* drafter row       l_q = l_p + N(0, sigma^2)   (sigma per workload)
* draft token       x ~ softmax(l_q / T), drawn by the Gumbel-max trick

All arithmetic is float32 in torch, rounded once to the storage dtype; rows
are independent across (b, k, j).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

QWEN_VOCAB = 152064
ZIPF_S = 1.1


@dataclass
class Workload:
    """One batch of verification inputs (tensors on one device)."""
    name: str
    B: int
    K: int
    gamma: int
    V: int
    dtype: torch.dtype
    p_logits: torch.Tensor            # [B, K, gamma+1, V]
    q_logits: torch.Tensor            # [B, K, gamma, V]
    drafts: torch.Tensor              # [B, K, gamma] int32
    temperature: float                # scalar temperature (used when temps is None)
    temps: Optional[torch.Tensor]     # [B] float32 per-sequence temperatures, or None
    seed: int = 0                     # Philox seed of the verification step
    identical: Sequence[int] = field(default_factory=list)  # b with q == p[:gamma]
    shared_q: bool = False            # q_logits is [B, gamma, V], shared by the K drafts

    def temps_list(self):
        if self.temps is None:
            return [float(self.temperature)] * self.B
        return [float(t) for t in self.temps.detach().cpu()]


def _zipf_prior(V: int, device) -> torch.Tensor:
    v = torch.arange(V, device=device, dtype=torch.float32)
    return -ZIPF_S * torch.log1p(v)


def _gumbel_argmax(rows_f32: torch.Tensor, inv_t: torch.Tensor, gen) -> torch.Tensor:
    """Draw one id per row from softmax(row * inv_t) (Gumbel-max)."""
    u = torch.rand(rows_f32.shape, generator=gen, device=rows_f32.device, dtype=torch.float32)
    g = -torch.log(-torch.log(u.clamp_min(1e-30)))
    return torch.argmax(rows_f32 * inv_t + g, dim=-1)


def generate(B: int, K: int, gamma: int, V: int, *, dtype=torch.bfloat16,
             p_sigma: float = 3.0, zipf: bool = True,
             q_sigma: Optional[torch.Tensor] = None,
             identical: Sequence[int] = (), temperature: float = 1.0,
             temps: Optional[torch.Tensor] = None, seed: int = 0,
             device="cpu", name: str = "custom", chunk_rows: int = 512,
             verify_seed: int = 0) -> Workload:
    """Build a workload.

    q_sigma: [B, K, gamma] drafter noise std (default 1.0 everywhere).
    identical: sequences b whose q rows are bitwise copies of p[b, :, :gamma].
    temps: optional [B] per-sequence temperatures (drafts use them).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    G1 = gamma + 1
    p = torch.empty((B, K, G1, V), dtype=dtype, device=device)
    q = torch.empty((B, K, gamma, V), dtype=dtype, device=device)
    prior = _zipf_prior(V, device) if zipf else None
    if q_sigma is None:
        q_sigma = torch.ones((B, K, gamma), dtype=torch.float32)
    q_sigma = q_sigma.to(device=device, dtype=torch.float32)
    if temps is not None:
        temps = temps.to(device=device, dtype=torch.float32)
        t_row = temps.view(B, 1, 1).expand(B, K, gamma).reshape(-1)
    else:
        t_row = torch.full((B * K * gamma,), float(temperature), device=device)
    ident = torch.zeros(B, dtype=torch.bool)
    for b in identical:
        ident[int(b)] = True
    ident_rows = ident.view(B, 1, 1).expand(B, K, gamma).reshape(-1).to(device)

    p_flat = p.view(-1, V)
    for r0 in range(0, p_flat.shape[0], chunk_rows):
        r1 = min(r0 + chunk_rows, p_flat.shape[0])
        x = torch.randn((r1 - r0, V), generator=gen, device=device, dtype=torch.float32)
        x.mul_(p_sigma)
        if prior is not None:
            x.add_(prior)
        p_flat[r0:r1] = x.to(dtype)

    q_flat = q.view(-1, V)
    sig_flat = q_sigma.reshape(-1)
    drafts = torch.empty((B * K * gamma,), dtype=torch.int64, device=device)
    # q row (b, k, j) pairs with p row (b, k, j): p row index = (b*K+k)*(gamma+1) + j
    nq = B * K * gamma
    for r0 in range(0, nq, chunk_rows):
        r1 = min(r0 + chunk_rows, nq)
        idx = torch.arange(r0, r1, device=device)
        bk, j = idx // gamma, idx % gamma
        prow = p_flat[bk * G1 + j].to(torch.float32)
        noise = torch.randn(prow.shape, generator=gen, device=device, dtype=torch.float32)
        qrow = prow + noise * sig_flat[r0:r1, None]
        qstore = qrow.to(dtype)
        same = ident_rows[r0:r1]
        if bool(same.any()):
            qstore[same] = p_flat[bk * G1 + j][same]
        q_flat[r0:r1] = qstore
        inv_t = (1.0 / t_row[r0:r1])[:, None]
        drafts[r0:r1] = _gumbel_argmax(qstore.to(torch.float32), inv_t, gen)
    return Workload(name=name, B=B, K=K, gamma=gamma, V=V, dtype=dtype, p_logits=p,
                    q_logits=q, drafts=drafts.view(B, K, gamma).to(torch.int32),
                    temperature=float(temperature), temps=temps, seed=int(verify_seed),
                    identical=[int(b) for b in identical])


def generate_shared(B: int, K: int, gamma: int, V: int, *, dtype=torch.bfloat16,
                    p_sigma: float = 3.0, zipf: bool = True,
                    q_sigma: Optional[torch.Tensor] = None, prefix_sigma: float = 0.5,
                    temperature: float = 1.0, temps: Optional[torch.Tensor] = None,
                    seed: int = 0, device="cpu", name: str = "shared-marginal",
                    chunk_rows: int = 256, verify_seed: int = 0) -> Workload:
    """Drafts from one denoising pass: the drafter exposes one marginal row per
    position, q[b, j] = base[b, j] + N(0, q_sigma[b, j]^2), and the K drafts are
    K independent samples from those marginals.  The verifier row at j = 0 sees
    only the prefix s, so it is the same row base[b, 0] for every draft; rows at
    j >= 1 see different draft prefixes: base[b, j] + N(0, prefix_sigma^2)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    G1 = gamma + 1
    prior = _zipf_prior(V, device) if zipf else None
    if q_sigma is None:
        q_sigma = torch.ones((B, gamma), dtype=torch.float32)
    q_sigma = q_sigma.to(device=device, dtype=torch.float32)
    if temps is not None:
        temps = temps.to(device=device, dtype=torch.float32)
    t_seq = temps if temps is not None else torch.full((B,), float(temperature), device=device)
    p = torch.empty((B, K, G1, V), dtype=dtype, device=device)
    q = torch.empty((B, gamma, V), dtype=dtype, device=device)
    drafts = torch.empty((B, K, gamma), dtype=torch.int64, device=device)
    for b in range(B):
        for j0 in range(0, G1, max(1, chunk_rows // max(K, 1))):
            j1 = min(G1, j0 + max(1, chunk_rows // max(K, 1)))
            base = torch.randn((j1 - j0, V), generator=gen, device=device, dtype=torch.float32)
            base.mul_(p_sigma)
            if prior is not None:
                base.add_(prior)
            rows = base.unsqueeze(0).expand(K, -1, -1).clone()
            noise = torch.randn(rows.shape, generator=gen, device=device, dtype=torch.float32)
            jj = torch.arange(j0, j1, device=device)
            rows += noise * prefix_sigma * (jj > 0).to(torch.float32)[None, :, None]
            p[b, :, j0:j1] = rows.to(dtype)
            for j in range(j0, min(j1, gamma)):
                qrow = base[j - j0] + torch.randn((V,), generator=gen, device=device) * q_sigma[b, j]
                qstore = qrow.to(dtype)
                q[b, j] = qstore
                logits = (qstore.to(torch.float32) / t_seq[b]).expand(K, V)
                drafts[b, :, j] = _gumbel_argmax(logits, torch.ones((), device=device), gen)
    return Workload(name=name, B=B, K=K, gamma=gamma, V=V, dtype=dtype, p_logits=p,
                    q_logits=q, drafts=drafts.to(torch.int32), temperature=float(temperature),
                    temps=temps, seed=int(verify_seed), shared_q=True)


def workload_shared(B: int = 32, K: int = 16, gamma: int = 32, V: int = QWEN_VOCAB,
                    device="cpu", seed: int = 55) -> Workload:
    """The large-window shape with drafts from one pass's marginals: drafter
    noise rising from 0.3 to 2.0 across the window, per-sequence temperatures
    in {0.6, 1.0}, verifier rows of different draft prefixes 0.5 apart."""
    g = torch.Generator(device="cpu")
    g.manual_seed(10_000 + seed)
    sj = 0.3 + 1.7 * torch.arange(gamma, dtype=torch.float32) / max(gamma - 1, 1)
    coin = torch.rand((B,), generator=g) < 0.5
    temps = torch.where(coin, torch.tensor(0.6), torch.tensor(1.0))
    return generate_shared(B, K, gamma, V, q_sigma=sj.expand(B, gamma).clone(), temps=temps,
                           seed=seed, device=device,
                           name="large-window shared-marginal B%d K%d g%d V%d bf16" % (B, K, gamma, V))


# --------------------------------------------------------------------------
# The five workloads (tiny exactness case, single stream, self-selection
# sweep, serving batch, large-window stress), each seeded by its index.
# --------------------------------------------------------------------------

CONFIGS = {
    1: dict(name="tiny-exact B1 K1 g4 V32 fp32", B=1, K=1, gamma=4, V=32),
    2: dict(name="single-stream B1 K1 g8 V152064 bf16", B=1, K=1, gamma=8, V=QWEN_VOCAB),
    3: dict(name="self-selection B8 K4 g16 V152064 bf16", B=8, K=4, gamma=16, V=QWEN_VOCAB),
    4: dict(name="serving B64 K8 g16 V152064 bf16", B=64, K=8, gamma=16, V=QWEN_VOCAB),
    5: dict(name="large-window B32 K16 g32 V152064 bf16", B=32, K=16, gamma=32, V=QWEN_VOCAB),
}


def config_shape(idx: int):
    c = CONFIGS[idx]
    return c["B"], c["K"], c["gamma"], c["V"]


def config_bytes(idx: int) -> int:
    """Bytes of the logit inputs of a workload."""
    B, K, G, V = config_shape(idx)
    elt = 4 if idx == 1 else 2
    return elt * V * B * K * (2 * G + 1)


def workload(idx: int, device="cpu", seed: Optional[int] = None,
             B: Optional[int] = None, V: Optional[int] = None) -> Workload:
    """Workload `idx` (1..5); B and V may be shrunk for fast tests, keeping
    every other parameter of the workload."""
    c = dict(CONFIGS[idx])
    B = c["B"] if B is None else B
    V = c["V"] if V is None else V
    K, G = c["K"], c["gamma"]
    seed = idx if seed is None else seed
    g = torch.Generator(device="cpu")
    g.manual_seed(10_000 + seed)
    if idx == 1:
        return generate(B, K, G, V, dtype=torch.float32, p_sigma=2.0, zipf=False,
                        q_sigma=torch.ones((B, K, G)), temperature=1.0, seed=seed,
                        device=device, name=c["name"])
    if idx == 2:
        return generate(B, K, G, V, dtype=torch.bfloat16, q_sigma=torch.full((B, K, G), 0.7),
                        temperature=1.0, seed=seed, device=device, name=c["name"])
    if idx == 3:
        sk = torch.rand((B, K, 1), generator=g) * 1.2 + 0.3
        ramp = 1.0 + torch.arange(G, dtype=torch.float32) / max(G - 1, 1)
        return generate(B, K, G, V, q_sigma=sk * ramp, temperature=0.7, seed=seed,
                        device=device, name=c["name"])
    if idx == 4:
        sbk = torch.rand((B, K, 1), generator=g) * 1.0 + 0.2
        n_same = int(round(0.3 * B))
        same = torch.randperm(B, generator=g)[:n_same].tolist()
        return generate(B, K, G, V, q_sigma=sbk.expand(B, K, G).clone(), identical=sorted(same),
                        temperature=1.0, seed=seed, device=device, name=c["name"])
    if idx == 5:
        sj = 0.3 + 1.7 * torch.arange(G, dtype=torch.float32) / max(G - 1, 1)
        coin = torch.rand((B,), generator=g) < 0.5
        temps = torch.where(coin, torch.tensor(0.6), torch.tensor(1.0))
        return generate(B, K, G, V, q_sigma=sj.expand(B, K, G).clone(), temps=temps,
                        temperature=1.0, seed=seed, device=device, name=c["name"])
    raise KeyError(idx)


def to_oracle_arrays(w: Workload, seqs: Optional[Sequence[int]] = None):
    """Host numpy copies of (a sample of) a workload in the oracle's formats:
    bf16 logits as raw uint16 words, float32 as is (q is None when the
    workload has no drafter rows)."""
    import numpy as np
    sl = slice(None) if seqs is None else list(seqs)
    def host(x):
        x = x[sl].detach().cpu().contiguous()
        return x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 else x.numpy()

    p = host(w.p_logits)
    q = None if w.q_logits is None else host(w.q_logits)     # none under greedy acceptance
    if w.shared_q and q is not None:    # the oracle takes the full layout: q broadcast over k
        q = np.ascontiguousarray(np.broadcast_to(q[:, None], (q.shape[0], w.K) + q.shape[1:]))
    d = w.drafts[sl].detach().cpu().numpy().astype(np.int32)
    t = np.asarray(w.temps_list(), dtype=np.float64)
    if seqs is not None:
        t = t[list(seqs)]
    return p, q, d, t
