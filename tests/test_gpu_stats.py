"""Statistical checks of the GPU outputs on the exactness workload
(B = 10^6 independent trials of one K=4, V=32 logit set).

- Emitted tokens are distributed as p~ (chi-square per position over the
  sequences that reach it; the bonus position against the target softmax of
  row K).  This is the lossless property of the modified rejection sampling
  ("修改的拒绝采样" and "1. 为什么无损" sections of the explainer pages), with
  p~ in place of the target distribution under RAPID's knowledge transfer.
- P(accept at i | reached i) = sum_v min(p~_v, q_v) (within 5 sigma).
- With equal acceptance at every position the mean number of emitted tokens is
  the explainer's 1 + a + a^2 + ... series, cut at K ("加速效果分析").
"""
import math

import numpy as np
import pytest
import scipy.stats
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def specv():
    import speculative_decoding_verification_specv_gb300 as m
    m.load(build_if_missing=True)
    return m


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("lam", [0.0, 0.25, 0.5])
def test_chi_square_and_acceptance(specv, mode, lam):
    w = workloads.WORKLOADS[5]
    x = workloads.make_inputs(w, DEV, lam=lam)
    tok, n = specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
                          x["u_resample"], x["lam"], mode=mode)
    tok = tok.cpu().numpy()
    n = n.cpu().numpy()
    zt0 = x["target_logits"][0].cpu()
    zq0 = x["draft_logits"][0].cpu()
    ptilde, q = oracle.rows(zt0, zq0, float(x["lam"][0]), mode)
    for j in range(w.K + 1):
        reached = n >= j
        obs = np.bincount(tok[reached, j], minlength=w.V).astype(np.float64)
        exp = ptilde[j] * reached.sum()
        keep = exp >= 5.0  # merge bins with tiny expectations into one
        o = np.append(obs[keep], obs[~keep].sum())
        e = np.append(exp[keep], exp[~keep].sum())
        if e[-1] == 0:
            o, e = o[:-1], e[:-1]
        stat, pval = scipy.stats.chisquare(o, e * o.sum() / e.sum())
        print(f"mode={mode} lam={lam} position {j}: n={reached.sum()} chi2={stat:.1f} p={pval:.3g}")
        assert pval > 1e-4, (j, stat, pval)
    for i in range(w.K):
        alpha = np.minimum(ptilde[i], q[i]).sum()
        reached = n >= i
        acc = (n[reached] > i).mean()
        sigma = math.sqrt(alpha * (1 - alpha) / reached.sum())
        assert abs(acc - alpha) < 5 * sigma, (i, acc, alpha, sigma)


def test_expected_tokens_series(specv):
    K, V, B = 4, 32, 1_000_000
    g = torch.Generator(device=DEV).manual_seed(77)
    zt1 = torch.randn(V, generator=g, device=DEV) * 1.5
    zq1 = torch.randn(V, generator=g, device=DEV) * 1.5
    zt = zt1.expand(B, K + 1, V).contiguous()
    zq = zq1.expand(B, K, V).contiguous()
    u = torch.rand((B, K, V), generator=g, device=DEV).clamp_min(1e-30)
    tok = torch.argmax(zq - torch.log(-torch.log(u)), dim=-1).to(torch.int32)
    del u
    ua = torch.rand((B, K), generator=g, device=DEV)
    ur = torch.rand((B,), generator=g, device=DEV)
    lam = torch.full((B,), 0.3, device=DEV)
    _, n = specv.verify(zt, zq, tok, ua, ur, lam, mode=0)
    n = n.cpu().numpy()
    ptilde, q = oracle.rows(zt[0].cpu(), zq[0].cpu(), float(lam[0]), 0)
    a = np.minimum(ptilde[0], q[0]).sum()
    mean = (1 - a ** (K + 1)) / (1 - a)
    ex2 = sum((2 * k + 1) * a ** k for k in range(K + 1))
    sd = math.sqrt((ex2 - mean * mean) / B)
    got = (n + 1).mean()
    print(f"alpha={a:.4f} mean emitted={got:.4f} series={mean:.4f} sd={sd:.2g}")
    assert abs(got - mean) < 5 * sd
