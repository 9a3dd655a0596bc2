"""Distribution-level checks of the CUDA path, independent of the oracle:
the first committed token of a step must follow the verifier's distribution
p_0 exactly.  Under the standard rule this holds for a single draft (K = 1;
"SpecDiff-2: Scaling Diffusion Drafter Alignment For Faster Speculative
Decoding", section 2).  Under greedy acceptance it holds for any K after
self-selection, since for every fixed draft token the committed token is
p-distributed (same page, section 5.2 and appendix B.4).  Each of 200 000
sequences repeats the same logits with its own draws; chi-square at a fixed
seed, alpha = 1e-3."""
import numpy as np
import pytest
import torch
from scipy import stats

from draft_verification_sdv_gb300 import binding as bd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bd.load(build=True)


def _batch(N, K, G, V, T, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    p1 = torch.randn((1, 1, G + 1, V), generator=g, device="cuda") * 1.5
    q1 = p1[:, :, :G] + torch.randn((1, 1, G, V), generator=g, device="cuda") * 1.0
    p = p1.expand(N, K, G + 1, V).contiguous()
    q = q1.expand(N, K, G, V).contiguous()
    probs_q = torch.softmax(q1[0, 0] / T, dim=-1)                       # [G, V]
    drafts = torch.stack([torch.multinomial(probs_q[j], N * K, replacement=True, generator=g)
                          for j in range(G)], dim=-1).view(N, K, G).to(torch.int32).contiguous()
    p0 = torch.softmax(p1[0, 0, 0].double() / T, dim=-1).cpu().numpy()
    return p, q, drafts, p0


def _first_token(out, drafts):
    L = out["accept_len"].long()
    sel = out["sel"].long()
    first_draft = drafts[torch.arange(drafts.shape[0], device="cuda"), sel, 0].long()
    return torch.where(L >= 1, first_draft, out["next_token"].long()).cpu().numpy()


def _chi2_ok(tokens, p0):
    V = len(p0)
    counts = np.bincount(tokens, minlength=V)
    expected = p0 * len(tokens)
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(expected[keep], expected[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    return stats.chisquare(obs, exp).pvalue


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_standard_rule_single_draft_commits_p(dtype):
    N, K, G, V, T = 200_000, 1, 3, 16, 0.9
    p, q, d, p0 = _batch(N, K, G, V, T, seed=90)
    p, q = p.to(dtype), q.to(dtype)
    if dtype == torch.bfloat16:                      # the distribution of the rounded logits
        p0 = torch.softmax(p[0, 0, 0].double() / T, dim=-1).cpu().numpy()
    v = bd.Verifier(N, K, G, V, dtype)
    out = v(p, q, d, temperature=T, seed=12345)
    v.sync()
    pv = _chi2_ok(_first_token(out, d), p0)
    assert pv > 1e-3, pv
    v.close()


def test_greedy_rule_with_selection_commits_p():
    N, K, G, V, T = 200_000, 2, 3, 16, 1.1
    p, q, d, p0 = _batch(N, K, G, V, T, seed=91)
    v = bd.Verifier(N, K, G, V, torch.float32, greedy=True)
    out = v(p, None, d, temperature=T, seed=777)
    v.sync()
    assert (out["sel"] >= 0).all()
    pv = _chi2_ok(_first_token(out, d), p0)
    assert pv > 1e-3, pv
    v.close()


def test_standard_rule_with_selection_departs_from_p():
    """The control that shows the test has teeth: under the standard rule,
    verifying only the best-scored of two drafts biases the first committed
    token away from p_0 (the counter-example of the oracle's pins), and the
    same chi-square rejects it."""
    N, K, G, V, T = 200_000, 2, 3, 16, 0.9
    p, q, d, p0 = _batch(N, K, G, V, T, seed=92)
    v = bd.Verifier(N, K, G, V, torch.float32)
    out = v(p, q, d, temperature=T, seed=4242)
    v.sync()
    pv = _chi2_ok(_first_token(out, d), p0)
    assert pv < 1e-6, pv
    v.close()
