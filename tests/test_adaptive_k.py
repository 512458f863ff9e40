"""Host-side draft-length policy (specv_choose_k and AdaptiveK), no GPU.

The policy maximises the expected tokens of one verify step, 1 + a + ... + a^K
(the speculative-decoding explainer's "加速效果分析" series, cut at the K
drafted tokens), per unit of step cost.  These tests pin it to the oracle's
own verify loop (tokens emitted per step, simulated), to brute force over K,
and to the limits the EAGLE explainer's "4. 草稿长度和接受率的权衡" describes:
a longer draft when acceptance is high, a shorter one when it is low.
"""
import math

import numpy as np
import pytest
import torch

import speculative_decoding_verification_specv_gb300 as specv


@pytest.fixture(scope="module")
def lib():
    return specv.load(build_if_missing=True)


def _rate(a, k, cd, cf, cv):
    tokens = sum(a ** j for j in range(k + 1))
    return tokens / (cf + k * (cd + cv))


@pytest.mark.parametrize("a", [0.0, 0.1, 0.35, 0.5, 0.62, 0.8, 0.9, 0.97, 1.0])
@pytest.mark.parametrize("costs", [(1.0, 10.0, 0.0), (0.5, 3.0, 0.2), (0.05, 1.0, 0.01),
                                   (2.0, 1.0, 0.0)])
def test_choose_k_is_the_brute_force_argmax(lib, a, costs):
    cd, cf, cv = costs
    k = specv.choose_k(a, cd, cf, cv, k_min=1, k_max=32)
    rates = [_rate(a, kk, cd, cf, cv) for kk in range(1, 33)]
    best = max(rates)
    assert rates[k - 1] == pytest.approx(best, rel=1e-12)
    # the smallest maximiser
    assert all(r < best * (1 - 1e-12) for r in rates[:k - 1])


def test_longer_drafts_for_higher_acceptance(lib):
    ks = [specv.choose_k(a, 0.3, 4.0, 0.05, 1, 64) for a in np.linspace(0.0, 0.99, 100)]
    assert all(x <= y for x, y in zip(ks, ks[1:]))
    assert ks[0] == 1 and ks[-1] > 8


def test_limits(lib):
    # no acceptance: every extra draft token only costs
    assert specv.choose_k(0.0, 1.0, 5.0, 0.0, 2, 9) == 2
    # certain acceptance, fixed cost larger than the per-token cost: the longest draft
    assert specv.choose_k(1.0, 0.5, 5.0, 0.1, 1, 12) == 12
    # free drafts and free verification per token: the rate only grows with K
    assert specv.choose_k(0.5, 0.0, 1.0, 0.0, 1, 7) == 7
    assert specv.choose_k(0.5, 1.0, 1.0, 0.0, 3, 3) == 3


@pytest.mark.parametrize("bad", [dict(alpha=-0.1), dict(alpha=1.5), dict(alpha=float("nan")),
                                 dict(k_min=0), dict(k_min=5, k_max=4), dict(k_max=5000),
                                 dict(cost_draft=-1.0), dict(cost_verify_fixed=0.0,
                                                             cost_draft=0.0)])
def test_bad_arguments(lib, bad):
    kw = dict(alpha=0.5, cost_draft=1.0, cost_verify_fixed=2.0, cost_verify_per_token=0.0,
              k_min=1, k_max=8)
    kw.update(bad)
    with pytest.raises(ValueError):
        specv.choose_k(**kw)


def test_policy_matches_the_oracles_measured_throughput(lib, oracle_mod):
    """Tokens emitted per step by the oracle's verify loop, averaged over many
    independent steps, for K = 1..6 with the same draft/target pair at every
    position: at every K the measured tokens per unit cost agree with the
    policy's objective at the oracle's exact acceptance probability, and the
    policy's K is the objective's (interior) maximiser."""
    V, B = 12, 30_000
    rng = np.random.default_rng(3)
    zt1 = rng.normal(0, 1.0, V).astype(np.float32)
    zq1 = (0.7 * zt1 + rng.normal(0, 1.5, V)).astype(np.float32)
    cd, cf, cv = 0.4, 2.0, 0.05
    objective = {}
    alpha = None
    for K in range(1, 7):
        zt = np.broadcast_to(zt1, (B, K + 1, V))
        zq = np.broadcast_to(zq1, (B, K, V))
        g = torch.Generator().manual_seed(100 + K)
        gum = -torch.log(-torch.log(torch.rand((B, K, V), generator=g).clamp_min(1e-30)))
        tok = torch.argmax(torch.from_numpy(zq.copy()) + gum, dim=-1).to(torch.int32)
        ua = torch.rand((B, K), generator=g)
        ur = torch.rand((B,), generator=g)
        r = oracle_mod.verify(zt, zq, tok, ua, ur, np.full(B, 0.3, np.float32))
        alpha = float(r.alpha[0, 0])
        emitted = (r.n_accepted + 1).astype(np.float64)
        cost = cf + K * (cd + cv)
        objective[K] = _rate(alpha, K, cd, cf, cv)
        sd = emitted.std() / math.sqrt(B) / cost
        assert abs(emitted.mean() / cost - objective[K]) < 5 * sd, (K, emitted.mean(), objective[K])
    k_policy = specv.choose_k(alpha, cd, cf, cv, 1, 6)
    assert 1 < k_policy < 6  # an interior optimum: the test separates it from the bounds
    assert objective[k_policy] == max(objective.values())


def test_adaptive_controller_follows_acceptance(lib):
    ctl = specv.AdaptiveK(cost_draft=0.3, cost_verify_fixed=4.0, cost_verify_per_token=0.05,
                          k_min=1, k_max=16, k_init=4, decay=0.5)
    assert ctl.k == 4
    for _ in range(20):
        k_hi = ctl.update(torch.full((8, 4), 0.95))
    assert k_hi == specv.choose_k(ctl.alpha, 0.3, 4.0, 0.05, 1, 16) and k_hi > 4
    for _ in range(20):
        k_lo = ctl.update(0.2)
    assert k_lo < k_hi and k_lo == specv.choose_k(ctl.alpha, 0.3, 4.0, 0.05, 1, 16)
    # NaN entries (sequences with invalid lambda) are ignored
    before = ctl.alpha
    ctl.update(torch.tensor([float("nan"), float("nan")]))
    assert ctl.alpha == before
    ctl.update(torch.tensor([0.5, float("nan")]))
    assert ctl.alpha == pytest.approx(0.5 * before + 0.5 * 0.5)
