"""Pins for the fp64 CPU oracle, checked against things other than itself.

Each test ties one part of the oracle to a closed form, a worked example
derived by hand from the pages (tests/golden/hand_cases.json), a mathematical
invariant, a library routine on a special case, or brute force on tiny inputs.
Sources: the RAPID explainer page ("2) 推理时知识迁移" mixture equation,
"3) 候选验证机制（伪代码）" loop), the speculative-decoding explainer page
("修改的拒绝采样", "加速效果分析") and the EAGLE explainer page
("1. 为什么无损": resample from max(0, p - q)).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


# --------------------------------------------------------------------------- softmax
def test_softmax_closed_form(oracle_mod):
    p = oracle_mod.softmax([0.0, math.log(2.0), math.log(3.0)])
    np.testing.assert_allclose(p, [1 / 6, 2 / 6, 3 / 6], rtol=0, atol=1e-15)


def test_softmax_large_logits_need_the_max_shift(oracle_mod):
    # exp(1000) overflows: only a max-shifted softmax gets [0.5, 0.5]
    np.testing.assert_array_equal(oracle_mod.softmax([1000.0, 1000.0]), [0.5, 0.5])
    np.testing.assert_allclose(oracle_mod.softmax([-1000.0, -1000.0 + math.log(3.0)]),
                               [0.25, 0.75], atol=1e-15)


def test_softmax_single_entry_and_library(oracle_mod):
    np.testing.assert_array_equal(oracle_mod.softmax([3.5]), [1.0])
    rng = np.random.default_rng(1)
    for V in (2, 7, 1000, 50_000):
        z = rng.normal(0, 4, V)
        np.testing.assert_allclose(oracle_mod.softmax(z), scipy.special.softmax(z),
                                   rtol=1e-12, atol=1e-300)


# --------------------------------------------------------------------------- mixtures
def test_mix_prob_special_values(oracle_mod):
    pt = np.array([0.5, 0.3, 0.2])
    pq = np.array([0.2, 0.2, 0.6])
    np.testing.assert_array_equal(oracle_mod.mix_prob(pt, pq, 0.0), pt)
    np.testing.assert_array_equal(oracle_mod.mix_prob(pt, pq, 1.0), pq)
    # lambda = 1/4 by hand: 0.75*pt + 0.25*pq
    np.testing.assert_allclose(oracle_mod.mix_prob(pt, pq, 0.25), [0.425, 0.275, 0.3],
                               atol=1e-15)


def test_mix_logit_closed_forms(oracle_mod):
    # V = 2: p~_0 = sigmoid(w_0 - w_1) with w = (1-l) z_t + l z_q
    zt = np.array([0.7, -1.1])
    zq = np.array([-0.4, 2.0])
    for lam in (0.0, 0.2, 0.5, 1.0):
        d = (1 - lam) * (zt[0] - zt[1]) + lam * (zq[0] - zq[1])
        got = oracle_mod.mix_logit(zt, zq, lam)
        np.testing.assert_allclose(got, [scipy.special.expit(d), scipy.special.expit(-d)],
                                   atol=1e-15)
    # lambda = 1/2: the logit mixture is the normalised geometric mean sqrt(p_t q)
    rng = np.random.default_rng(2)
    zt = rng.normal(0, 2, 64)
    zq = rng.normal(0, 2, 64)
    g = np.sqrt(scipy.special.softmax(zt) * scipy.special.softmax(zq))
    np.testing.assert_allclose(oracle_mod.mix_logit(zt, zq, 0.5), g / g.sum(), rtol=1e-12)


def test_rows_sum_to_one(oracle_mod):
    w = workloads.WORKLOADS[3].scaled(B=2, V=4099)
    x = workloads.make_inputs(w)
    for mode in (oracle_mod.PROB_MIX, oracle_mod.LOGIT_MIX):
        for b in range(2):
            pt, q = oracle_mod.rows(x["target_logits"][b], x["draft_logits"][b],
                                    float(x["lam"][b]), mode)
            np.testing.assert_allclose(pt.sum(axis=1), 1.0, atol=1e-12)
            np.testing.assert_allclose(q.sum(axis=1), 1.0, atol=1e-12)
            assert (pt >= 0).all() and (q >= 0).all()


def test_lambda_zero_is_plain_target(oracle_mod):
    w = workloads.WORKLOADS[1].scaled(V=257)
    x = workloads.make_inputs(w)
    for mode in (oracle_mod.PROB_MIX, oracle_mod.LOGIT_MIX):
        pt, q = oracle_mod.rows(x["target_logits"][0], x["draft_logits"][0], 0.0, mode)
        for i in range(w.K + 1):
            ref = scipy.special.softmax(x["target_logits"][0, i].double().numpy())
            np.testing.assert_allclose(pt[i], ref, rtol=1e-12)
        for i in range(w.K):
            ref = scipy.special.softmax(x["draft_logits"][0, i].double().numpy())
            np.testing.assert_allclose(q[i], ref, rtol=1e-12)


# --------------------------------------------------------------------------- inverse CDF
def test_inverse_cdf_hand_cases(oracle_mod):
    w = [1.0, 2.0, 3.0, 0.0]       # CDF boundaries 1/6, 1/2, 1
    assert oracle_mod.sample_inverse_cdf(w, 0.0)[0] == 0
    assert oracle_mod.sample_inverse_cdf(w, 0.1)[0] == 0
    assert oracle_mod.sample_inverse_cdf(w, 0.2)[0] == 1
    assert oracle_mod.sample_inverse_cdf(w, 0.49)[0] == 1
    assert oracle_mod.sample_inverse_cdf(w, 0.51)[0] == 2
    assert oracle_mod.sample_inverse_cdf(w, 0.999999)[0] == 2
    assert oracle_mod.sample_inverse_cdf([0.0, 0.0], 0.5)[0] == -1
    # u = 1 leaves no prefix strictly above u*W: the last positive weight is taken
    idx, fb, _ = oracle_mod.sample_inverse_cdf([0.5, 0.25, 0.0], 1.0)
    assert idx == 1 and fb
    # the margin is the distance of u to the nearest boundary C_k / W
    _, _, m = oracle_mod.sample_inverse_cdf(w, 0.49)
    assert m == pytest.approx(0.01, abs=1e-12)


def test_inverse_cdf_maps_uniform_grid_to_the_distribution(oracle_mod):
    # Midpoints of N equal cells: each index is hit N*w_v/W times up to one
    # cell per boundary.  Zero-weight indices are never hit.
    rng = np.random.default_rng(3)
    w = rng.random(13) * (rng.random(13) > 0.3)
    N = 20000
    counts = np.zeros(13)
    for k in range(N):
        counts[oracle_mod.sample_inverse_cdf(w, (k + 0.5) / N)[0]] += 1
    assert (counts[w == 0] == 0).all()
    np.testing.assert_allclose(counts / N, w / w.sum(), atol=1.0 / N + 1e-12)


# --------------------------------------------------------------------------- worked examples
def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_examples(oracle_mod, case):
    pt = np.array(case["p_t"], np.float64)
    q = np.array(case["q"], np.float64)
    K = q.shape[0]
    zt = np.log(pt).astype(np.float32)[None]
    zq = np.log(q).astype(np.float32)[None]
    mode = oracle_mod.PROB_MIX if case["mode"] == "prob" else oracle_mod.LOGIT_MIX
    r = oracle_mod.verify(zt, zq, np.array([case["tokens"]], np.int32),
                          np.array([case["u_accept"]], np.float32),
                          np.array([case["u_resample"]], np.float32),
                          np.array([case["lam"]], np.float32), mode=mode)
    assert r.tokens[0].tolist() == case["expect_tokens"]
    assert int(r.n_accepted[0]) == case["expect_n"]
    if "expect_ratio" in case:
        np.testing.assert_allclose(r.ratio[0], case["expect_ratio"], rtol=2e-6)
        np.testing.assert_allclose(r.alpha[0], case["expect_alpha"], rtol=2e-6)


# --------------------------------------------------------------------------- exactness
def _lattice(N, g):
    i = np.arange(N, dtype=np.float64)
    return ((i + 0.5) / N).astype(np.float32), (np.mod(i * g + 0.5, N) / N).astype(np.float32)


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("lam", [0.0, 0.3, 0.8])
def test_output_distribution_is_ptilde_by_quadrature(oracle_mod, mode, lam):
    """Brute force over the draft token and a rank-1 lattice of uniform pairs.

    The token emitted at position 0 must be distributed as p~_0 (accept with
    min(1, p~/q), else resample max(0, p~ - q)), and the bonus token, given
    that the draft passed, as the target softmax of row 1.
    """
    rng = np.random.default_rng(7 + mode)
    V = 5
    zt = rng.normal(0, 1.5, (1, 2, V)).astype(np.float32)
    zq = rng.normal(0, 1.5, (1, 1, V)).astype(np.float32)
    ptilde, q = oracle_mod.rows(zt[0], zq[0], lam, mode)
    N = 1 << 15
    ua, ur = _lattice(N, 20261)          # generator close to N / golden ratio, odd
    dist0 = np.zeros(V)
    bonus = np.zeros(V)
    bonus_w = 0.0
    for x in range(V):
        r = oracle_mod.verify(np.broadcast_to(zt, (N, 2, V)), np.broadcast_to(zq, (N, 1, V)),
                              np.full((N, 1), x, np.int32), ua[:, None], ur,
                              np.full(N, lam, np.float32), mode=mode, diagnostics=False)
        t0 = r.tokens[:, 0]
        dist0 += q[0, x] * np.bincount(t0, minlength=V) / N
        acc = r.n_accepted == 1
        bonus += q[0, x] * np.bincount(r.tokens[acc, 1], minlength=V) / N
        bonus_w += q[0, x] * acc.mean()
    np.testing.assert_allclose(dist0, ptilde[0], atol=2e-3)
    np.testing.assert_allclose(bonus / bonus_w, scipy.special.softmax(zt[0, 1].astype(np.float64)),
                               atol=2e-3)


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
def test_chi_square_and_acceptance_rate_monte_carlo(oracle_mod, mode):
    """Monte Carlo with the exactness workload's recipe at V = 8, K = 2."""
    w = workloads.WORKLOADS[5].scaled(B=200_000, K=2, V=8)
    x = workloads.make_inputs(w, lam=0.4)
    r = oracle_mod.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                          x["u_accept"], x["u_resample"], x["lam"], mode=mode)
    ptilde, q = oracle_mod.rows(x["target_logits"][0], x["draft_logits"][0], float(x["lam"][0]),
                                mode)
    n = r.n_accepted
    for j in range(w.K + 1):
        reached = n >= j
        obs = np.bincount(r.tokens[reached, j], minlength=w.V)
        exp = ptilde[j] * reached.sum()
        stat, pval = scipy.stats.chisquare(obs, exp)
        assert pval > 1e-4, (j, stat, pval)
    # P(accept at i | reached i) = sum_v min(p~, q) = 1 - TV(p~, q)
    for i in range(w.K):
        alpha = r.alpha[0, i]
        assert alpha == pytest.approx(1 - 0.5 * np.abs(ptilde[i] - q[i]).sum(), abs=1e-12)
        reached = n >= i
        acc = (n[reached] > i).mean()
        sigma = math.sqrt(alpha * (1 - alpha) / reached.sum())
        assert abs(acc - alpha) < 5 * sigma, (i, acc, alpha, sigma)


def test_expected_tokens_formula_truncated(oracle_mod):
    """With the same alpha at every position, the mean number of emitted tokens
    is 1 + a + ... + a^K = (1 - a^(K+1)) / (1 - a) (the explainer's
    1/(1 - r) series, cut at the K drafted tokens)."""
    K, V, B = 4, 16, 100_000
    rng = np.random.default_rng(11)
    zt1 = rng.normal(0, 1.5, V).astype(np.float32)
    zq1 = rng.normal(0, 1.5, V).astype(np.float32)
    zt = np.broadcast_to(zt1, (B, K + 1, V))
    zq = np.broadcast_to(zq1, (B, K, V))
    g = torch.Generator().manual_seed(5)
    gum = -torch.log(-torch.log(torch.rand((B, K, V), generator=g).clamp_min(1e-30)))
    tok = torch.argmax(torch.from_numpy(zq.copy()) + gum, dim=-1).to(torch.int32)
    ua = torch.rand((B, K), generator=g)
    ur = torch.rand((B,), generator=g)
    r = oracle_mod.verify(zt, zq, tok, ua, ur, np.full(B, 0.3, np.float32))
    a = r.alpha[0, 0]
    assert np.allclose(r.alpha[0], a)
    emitted = r.n_accepted + 1
    mean = (1 - a ** (K + 1)) / (1 - a)
    ex2 = sum((2 * k + 1) * a ** k for k in range(K + 1))  # E[m^2], m = tokens emitted
    sd = math.sqrt((ex2 - mean * mean) / B)
    assert abs(emitted.mean() - mean) < 5 * sd


# --------------------------------------------------------------------------- special cases
def test_identical_draft_and_target_accepts_everything(oracle_mod):
    w = workloads.WORKLOADS[4].scaled(B=8, V=3001)
    x = workloads.make_inputs(w)
    h = w.B // 2
    for mode in (0, 1):
        for lam in (0.0, 0.2):
            r = oracle_mod.verify(x["target_logits"][h:], x["draft_logits"][h:],
                                  x["draft_tokens"][h:], x["u_accept"][h:],
                                  x["u_resample"][h:], np.full(w.B - h, lam, np.float32),
                                  mode=mode)
            assert (r.n_accepted == w.K).all()
            assert (r.flags & oracle_mod.FLAG_BONUS).all()


def test_lambda_one_prob_mode_accepts_everything(oracle_mod):
    w = workloads.WORKLOADS[3].scaled(B=4, V=2049)
    x = workloads.make_inputs(w, lam=1.0)
    r = oracle_mod.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                          x["u_accept"], x["u_resample"], x["lam"], mode=0)
    assert (r.n_accepted == w.K).all()


def test_zero_uniform_accepts_unless_ptilde_is_zero(oracle_mod):
    w = workloads.WORKLOADS[1].scaled(B=16, V=101)
    x = workloads.make_inputs(w)
    ua = torch.zeros_like(x["u_accept"])
    r = oracle_mod.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"], ua,
                          x["u_resample"], x["lam"])
    assert (r.n_accepted == w.K).all()
    # p~(x) = 0 with q(x) > 0 (logits of -inf-like size) rejects even at u = 0
    zt = np.array([[[-200.0, 0.0], [0.0, 0.0]]], np.float32)
    zq = np.array([[[0.0, 0.0]]], np.float32)
    r = oracle_mod.verify(zt, zq, np.array([[0]], np.int32), np.zeros((1, 1), np.float32),
                          np.array([0.5], np.float32), np.array([0.0], np.float32))
    # p~(x) = e^-200 / (1 + e^-200) > 0 in fp64, so this still accepts
    assert r.n_accepted[0] == 1
    # push the target probability of x to an exact zero
    zt[0, 0, 0] = -1e30
    r = oracle_mod.verify(zt, zq, np.array([[0]], np.int32), np.zeros((1, 1), np.float32),
                          np.array([0.5], np.float32), np.array([0.0], np.float32))
    assert r.n_accepted[0] == 0 and r.tokens[0].tolist() == [1, -1]


def test_decision_margins_hand_case(oracle_mod):
    """The margins that the GPU parity tests use to tell a rounding-order tie
    from a real mismatch: accept_margin is the smallest |u_i - min(1, ratio_i)|
    over the positions actually decided (none after the first rejection), and
    cdf_margin the smallest |u - C_v / W| over the boundaries of the CDF the
    token was drawn from."""
    # p_t rows (0.25, 0.75), (0.5, 0.5), bonus row (0.5, 0.5); q rows (0.5, 0.5);
    # lambda = 0; both drafts are token 0
    zt = np.log(np.array([[[0.25, 0.75], [0.5, 0.5], [0.5, 0.5]]])).astype(np.float32)
    zq = np.log(np.array([[[0.5, 0.5], [0.5, 0.5]]])).astype(np.float32)
    tok = np.array([[0, 0]], np.int32)
    lam = np.array([0.0], np.float32)
    # position 0: ratio 0.5, u = 0.6 rejects; position 1 (u = 0.98, ratio 1) is
    # never decided, so its distance 0.02 does not count.  Residual (0, 0.25):
    # boundaries 0 and 1, u = 0.3 -> token 1 at distance 0.3.
    r = oracle_mod.verify(zt, zq, tok, np.array([[0.6, 0.98]], np.float32),
                          np.array([0.3], np.float32), lam)
    assert r.n_accepted.tolist() == [0] and r.tokens.tolist() == [[1, -1, -1]]
    assert r.accept_margin[0] == pytest.approx(0.1, abs=1e-6)
    assert r.cdf_margin[0] == pytest.approx(0.3, abs=1e-6)
    # both accepted (distances 0.1 and 0.02); bonus from (0.5, 0.5): boundaries
    # 0.5 and 1, u = 0.3 -> token 0 at distance 0.2
    r = oracle_mod.verify(zt, zq, tok, np.array([[0.4, 0.98]], np.float32),
                          np.array([0.3], np.float32), lam)
    assert r.n_accepted.tolist() == [2] and r.tokens.tolist() == [[0, 0, 0]]
    assert r.accept_margin[0] == pytest.approx(0.02, abs=1e-6)
    assert r.cdf_margin[0] == pytest.approx(0.2, abs=1e-6)


def test_seq_range_and_threads_do_not_change_results(oracle_mod):
    w = workloads.WORKLOADS[3].scaled(B=12, V=999)
    x = workloads.make_inputs(w)
    a = oracle_mod.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                          x["u_accept"], x["u_resample"], x["lam"], threads=1)
    b = oracle_mod.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                          x["u_accept"], x["u_resample"], x["lam"], threads=5)
    np.testing.assert_array_equal(a.tokens, b.tokens)
    np.testing.assert_array_equal(a.n_accepted, b.n_accepted)
    np.testing.assert_array_equal(a.ratio, b.ratio)


# --------------------------------------------------------------------------- greedy
# The greedy clause of the EAGLE explainer ("核心思路", step 3): a draft token
# equal to the target's most likely token is accepted.  Read with RAPID's
# mixture as: accept x_i iff x_i = argmax_v w_v, w = (1 - lambda) z_t + lambda z_q
# (in double precision); emit the argmax at the first mismatch, the argmax of
# target row K if all match.

def _np_greedy(zt, zq, tok, lam):
    """Independent restatement for inputs on which every fp32 operation of w is
    exact (small integers, dyadic lambda): w in float64, numpy's argmax (first
    index among equal maxima)."""
    B, K1, V = zt.shape
    K = K1 - 1
    out_t = np.full((B, K + 1), -1, np.int32)
    out_n = np.zeros(B, np.int32)
    for b in range(B):
        n = K
        for i in range(K):
            w = zt[b, i].astype(np.float64) + lam[b] * (zq[b, i].astype(np.float64) -
                                                         zt[b, i].astype(np.float64))
            a = int(np.argmax(w))
            if a != tok[b, i]:
                n, t = i, a
                break
            out_t[b, i] = tok[b, i]
        if n == K:
            t = int(np.argmax(zt[b, K]))
        out_t[b, n] = t
        out_n[b] = n
    return out_t, out_n


def test_greedy_lambda_zero_is_the_target_argmax(oracle_mod):
    rng = np.random.default_rng(7)
    for V in (1, 2, 17, 1000):
        zt = rng.normal(0, 3, V).astype(np.float32)
        zq = rng.normal(0, 3, V).astype(np.float32)
        assert oracle_mod.greedy_argmax(zt, zq, 0.0) == int(np.argmax(zt))
        assert oracle_mod.greedy_argmax(zt, None, 0.7) == int(np.argmax(zt))


def test_greedy_exact_mixtures_match_an_independent_restatement(oracle_mod):
    rng = np.random.default_rng(11)
    for lam in (0.0, 0.25, 0.5, 0.75, 1.0):
        B, K, V = 40, 4, 9
        zt = rng.integers(-8, 9, (B, K + 1, V)).astype(np.float32)
        zq = rng.integers(-8, 9, (B, K, V)).astype(np.float32)
        lams = np.full(B, lam, np.float32)
        # half the drafts follow the mixture's argmax, so prefixes get accepted
        tok = rng.integers(0, V, (B, K)).astype(np.int32)
        for b in range(0, B, 2):
            for i in range(K):
                w = zt[b, i] + lam * (zq[b, i] - zt[b, i])
                tok[b, i] = int(np.argmax(w))
        res = oracle_mod.verify_greedy(zt, zq, tok, lams, threads=1)
        et, en = _np_greedy(zt, zq, tok, lams)
        np.testing.assert_array_equal(res.n_accepted, en)
        np.testing.assert_array_equal(res.tokens, et)
        assert (res.n_accepted[0::2] == K).all()


def test_greedy_hand_case(oracle_mod):
    # K = 3, V = 4, lambda = 0.5.  Rows (w = mean of the two logit rows):
    #   i=0: zt [0,4,0,0], zq [0,2,0,0] -> w [0,3,0,0], argmax 1 = x_0: accept
    #   i=1: zt [1,0,0,3], zq [5,0,0,1] -> w [3,0,0,2], argmax 0 = x_1: accept
    #   i=2: zt [0,0,2,2], zq [0,0,0,2] -> w [0,0,1,2], argmax 3 != x_2 = 2: stop
    # so n = 2 and the emitted token is 3.
    zt = np.array([[[0, 4, 0, 0], [1, 0, 0, 3], [0, 0, 2, 2], [9, 0, 0, 0]]], np.float32)
    zq = np.array([[[0, 2, 0, 0], [5, 0, 0, 1], [0, 0, 0, 2]]], np.float32)
    tok = np.array([[1, 0, 2]], np.int32)
    res = oracle_mod.verify_greedy(zt, zq, tok, np.array([0.5], np.float32))
    assert res.n_accepted.tolist() == [2]
    assert res.tokens.tolist() == [[1, 0, 3, -1]]
    # with x_2 = 3 every draft matches: bonus = argmax of target row K = 0
    res = oracle_mod.verify_greedy(zt, zq, np.array([[1, 0, 3]], np.int32),
                                   np.array([0.5], np.float32))
    assert res.n_accepted.tolist() == [3] and res.tokens.tolist() == [[1, 0, 3, 0]]


def test_greedy_ties_masked_drafts_and_invalid_inputs(oracle_mod):
    # equal maxima: the smallest index
    assert oracle_mod.greedy_argmax(np.array([1, 7, 7, 7], np.float32), None, 0.0) == 1
    # a draft logit of -inf removes the entry from the mixture
    zt = np.array([0, 0, 0, 5], np.float32)
    zq = np.array([0, 1, 0, -np.inf], np.float32)
    assert oracle_mod.greedy_argmax(zt, zq, 0.25) == 1
    # invalid token or lambda: everything -1
    B, K, V = 3, 2, 5
    zt = np.zeros((B, K + 1, V), np.float32)
    zq = np.zeros((B, K, V), np.float32)
    tok = np.zeros((B, K), np.int32)
    tok[1, 1] = V
    lam = np.array([0.1, 0.1, 1.5], np.float32)
    res = oracle_mod.verify_greedy(zt, zq, tok, lam)
    assert res.n_accepted.tolist() == [2, -1, -1]
    assert (res.tokens[1:] == -1).all()
    # all-equal rows: every argmax is 0, so drafts of 0 are all accepted
    assert res.tokens[0].tolist() == [0, 0, 0]


def test_greedy_takes_the_exact_argmax_where_fp32_orders_the_other_way(oracle_mod):
    """Two entries whose mixed logits differ by 6.4e-8: in exact rational
    arithmetic entry 1 is larger, while z_t + lambda (z_q - z_t) formed in fp32
    (one rounded subtraction, one fused multiply-add) makes entry 0 larger.
    The oracle follows the mathematics, not the fp32 rounding."""
    from fractions import Fraction as Fr
    lam = np.float32(0.2884209)
    zt = np.array([1.0595762729644775, 3.342172622680664], np.float32)
    zq = np.array([1.8662627935409546, -3.765256643295288], np.float32)
    L = Fr(float(lam))
    exact = [(1 - L) * Fr(float(zt[v])) + L * Fr(float(zq[v])) for v in range(2)]
    assert exact[1] > exact[0] and float(exact[1] - exact[0]) > 6e-8
    # the fp32 path: each operation exact in fp64 here, then rounded once to fp32
    d = np.float32(zq - zt)
    w32 = [np.float32(float(Fr(float(lam)) * Fr(float(d[v])) + Fr(float(zt[v])))) for v in range(2)]
    assert w32[0] > w32[1]
    idx, gap = oracle_mod.greedy_argmax(zt, zq, lam, with_gap=True)
    assert idx == 1
    # the relative gap is the exact difference over the largest |logit| (3.765...)
    assert gap == pytest.approx(float((exact[1] - exact[0]) / Fr(float(abs(zq[1])))), rel=1e-6)
    assert gap < 2.0 ** -20  # inside the tie band of the GPU parity tests


def test_greedy_tie_margin_covers_the_decided_rows_only(oracle_mod):
    # K = 2, V = 3, lambda = 0: w = z_t.  Row 0 [0, 4, 1]: gap 3, max |z| 4
    # (both rows count, so A = max(|z_t|, |z_q|) = 8 from z_q) -> 3/8.
    # Row 1 [2, 2, 0] is an exact tie (gap 0) but is read only when x_0 = 1.
    zt = np.array([[[0, 4, 1], [2, 2, 0], [5, 0, 0]]], np.float32)
    zq = np.array([[[8, 0, 0], [0, 0, 1]]], np.float32)
    lam = np.array([0.0], np.float32)
    res = oracle_mod.verify_greedy(zt, zq, np.array([[0, 0]], np.int32), lam)
    assert res.n_accepted.tolist() == [0] and res.tokens.tolist() == [[1, -1, -1]]
    assert res.tie_margin[0] == pytest.approx(3 / 8)
    res = oracle_mod.verify_greedy(zt, zq, np.array([[1, 0]], np.int32), lam)
    assert res.n_accepted.tolist() == [2] and res.tokens.tolist() == [[1, 0, 0]]
    assert res.tie_margin[0] == 0.0
    # only the bonus row left: nothing of rounding to report
    res = oracle_mod.verify_greedy(zt[:, 1:], zq[:, 1:], np.array([[0]], np.int32), lam)
    assert res.n_accepted.tolist() == [1] and res.tie_margin[0] == 0.0


# ------------------------------------------------------------- masked logits
# Reading for -inf logits in the logit mixture (1 - lambda) z_t + lambda z_q:
# a -inf entry of positive weight gives -inf; a zero-weight term drops out.

def test_masked_logit_mixture_rule(oracle_mod):
    ninf = float("-inf")
    assert oracle_mod.mix_logit_entry(ninf, 1.5, 1.0) == 1.5
    assert oracle_mod.mix_logit_entry(ninf, 1.5, 0.5) == ninf
    assert oracle_mod.mix_logit_entry(ninf, 1.5, 0.0) == ninf
    assert oracle_mod.mix_logit_entry(2.0, ninf, 0.0) == 2.0
    assert oracle_mod.mix_logit_entry(2.0, ninf, 0.25) == ninf
    assert oracle_mod.mix_logit_entry(2.0, ninf, 1.0) == ninf
    assert oracle_mod.mix_logit_entry(ninf, ninf, 0.0) == ninf
    assert oracle_mod.mix_logit_entry(2.0, 4.0, 0.25) == 2.5
    # softmax of the mixed row: masked entries get probability 0, the rest the
    # closed form (lambda = 1/2: mixed entries [0, ln 3] -> weights [1, 3])
    zt = np.array([0.0, ninf, 2.0 * np.log(3.0), 0.0])
    zq = np.array([0.0, 5.0, 0.0, ninf])
    p = oracle_mod.mix_logit(zt, zq, 0.5)
    np.testing.assert_allclose(p, [0.25, 0.0, 0.75, 0.0], rtol=0, atol=1e-15)
    p0 = oracle_mod.mix_logit(zt, zq, 0.0)  # lambda = 0: the target softmax
    np.testing.assert_allclose(p0, oracle_mod.softmax(zt), rtol=0, atol=1e-15)
    p1 = oracle_mod.mix_logit(zt, zq, 1.0)  # lambda = 1: the draft softmax
    np.testing.assert_allclose(p1, oracle_mod.softmax(zq), rtol=0, atol=1e-15)


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
def test_draft_token_masked_in_the_draft_row(oracle_mod, mode):
    """q(x) = 0: the ratio is +inf, so x is accepted whenever p~(x) > 0, and
    rejected when p~(x) = 0 too (then the residual is drawn)."""
    ninf = np.float32(-np.inf)
    zt = np.array([[[0.0, 2.0, 1.0], [0.0, 0.0, 0.0]]], np.float32)
    zq = np.array([[[1.0, ninf, 0.0]]], np.float32)
    tok = np.array([[1]], np.int32)
    ua = np.array([[0.999]], np.float32)
    ur = np.array([0.5], np.float32)
    # lambda = 0.3: p~(1) > 0 in probability mode (0.7 p_t(1)); in logit mode
    # the mixed entry is -inf (the draft's mask has weight 0.3), so p~(1) = 0
    res = oracle_mod.verify(zt, zq, tok, ua, ur, np.array([0.3], np.float32), mode=mode)
    if mode == 0:
        assert res.n_accepted.tolist() == [1] and res.ratio[0, 0] == np.inf
    else:
        assert res.n_accepted.tolist() == [0] and res.ratio[0, 0] == 0.0
        # residual max(0, p~ - q): p~ = softmax([0.3, -inf, 0.7]) puts 0.599 on
        # entry 2, q = softmax([1, -inf, 0]) puts 0.269 there (and more than p~
        # on entry 0), so the residual lives on entry 2 alone
        assert res.tokens.tolist() == [[2, -1]]
    # lambda = 0 in logit mode: the draft's mask has weight 0, p~ = p_t, accept
    res = oracle_mod.verify(zt, zq, tok, ua, ur, np.array([0.0], np.float32), mode=mode)
    assert res.n_accepted.tolist() == [1]
    # lambda = 1 in probability mode: p~ = q, p~(1) = 0: reject
    res = oracle_mod.verify(zt, zq, tok, ua, ur, np.array([1.0], np.float32), mode=mode)
    assert res.n_accepted.tolist() == [0]
