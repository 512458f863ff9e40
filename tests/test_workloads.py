"""The seeded input generators against the recipes they state (CPU).

The five benchmark workloads are synthetic stand-ins: Gaussian logits of the
stated scale and draft/target correlation, per-sequence lambda where stated,
the drafted-equals-target half of the batched workload, one broadcast row set
for the short-row workload, and draft tokens drawn from the draft softmax.
These tests check each recipe on reduced batch and vocabulary sizes (the
recipes do not depend on the sizes) against the statistics it implies.
"""
import numpy as np
import pytest
import torch

import workloads

W = workloads.WORKLOADS


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _slope_and_residual(zt, zq):
    """Least-squares fit zq = a * zt + r over all entries: (a, std(r))."""
    x, y = zt.ravel(), zq.ravel()
    a = float(np.dot(x, y) / np.dot(x, x))
    return a, float(np.std(y - a * x))


def test_correlated_recipe_scale_slope_and_noise():
    # workload 1: z_t ~ N(0, 2^2); z_q = 0.8 z_t + N(0, 1)
    x = workloads.make_inputs(W[1].scaled(B=32, V=4096))
    zt, zq = _np(x["target_logits"]), _np(x["draft_logits"])
    assert abs(zt.mean()) < 0.02 and zt.std() == pytest.approx(2.0, rel=0.01)
    a, r = _slope_and_residual(zt[:, :-1], zq)
    assert a == pytest.approx(0.8, abs=0.005) and r == pytest.approx(1.0, rel=0.01)
    assert x["lam"].tolist() == pytest.approx([0.3] * 32)


def test_rho_recipe_per_sequence_correlation_and_equal_variance():
    # workload 3: rho_b ~ U(0.5, 0.95); z_q = rho z_t + sqrt(1 - rho^2) 3 eps; bf16
    x = workloads.make_inputs(W[3].scaled(B=64, V=20000))
    assert x["target_logits"].dtype == torch.bfloat16
    zt, zq = _np(x["target_logits"]), _np(x["draft_logits"])
    rhos = np.array([np.corrcoef(zt[b, :-1].ravel(), zq[b].ravel())[0, 1] for b in range(64)])
    assert rhos.min() > 0.5 - 0.02 and rhos.max() < 0.95 + 0.02
    assert rhos.max() - rhos.min() > 0.3  # spread over the interval, not one value
    assert zt.std() == pytest.approx(3.0, rel=0.01) and zq.std() == pytest.approx(3.0, rel=0.01)
    lam = x["lam"].numpy()
    assert lam.min() >= 0.0 and lam.max() < 0.5 and lam.max() - lam.min() > 0.3


def test_half_equal_recipe():
    # workload 4: as workload 1's recipe (scale 3, slope 0.85, noise 1) for b < B/2,
    # drafted rows equal to the target rows for b >= B/2; fp32
    w = W[4].scaled(B=16, V=8192)
    x = workloads.make_inputs(w)
    zt, zq = x["target_logits"], x["draft_logits"]
    assert zt.dtype == torch.float32
    assert torch.equal(zq[8:], zt[8:, :w.K])
    assert not torch.equal(zq[:8], zt[:8, :w.K])
    a, r = _slope_and_residual(_np(zt[:8, :-1]), _np(zq[:8]))
    assert a == pytest.approx(0.85, abs=0.005) and r == pytest.approx(1.0, rel=0.01)
    assert _np(zt).std() == pytest.approx(3.0, rel=0.01)


def test_broadcast_recipe_one_row_set_for_every_sequence():
    # workload 5: one z_t [K+1][V] and one independent z_q [K][V], N(0, 1.5^2)
    w = W[5].scaled(B=500, V=4096)
    x = workloads.make_inputs(w)
    zt, zq = x["target_logits"], x["draft_logits"]
    assert torch.equal(zt, zt[:1].expand_as(zt)) and torch.equal(zq, zq[:1].expand_as(zq))
    t1, q1 = _np(zt[0]), _np(zq[0])
    assert t1.std() == pytest.approx(1.5, rel=0.03) and q1.std() == pytest.approx(1.5, rel=0.03)
    assert abs(np.corrcoef(t1[:-1].ravel(), q1.ravel())[0, 1]) < 0.03
    # every sequence draws its own tokens and uniforms
    assert len(set(map(tuple, x["draft_tokens"].tolist()))) > 100


def test_draft_tokens_follow_the_draft_softmax():
    """Gumbel-max draws against the fp64 softmax of the stored draft rows, per
    position: a chi-square test over 200 000 independent draws of one row set."""
    from scipy import stats
    w = W[5].scaled(B=200_000)
    x = workloads.make_inputs(w)
    zq = _np(x["draft_logits"][0])
    tok = x["draft_tokens"].numpy()
    for i in range(w.K):
        p = np.exp(zq[i] - zq[i].max())
        p /= p.sum()
        counts = np.bincount(tok[:, i], minlength=w.V)
        expected = p * w.B
        keep = expected >= 5  # merge the small bins into one
        obs = np.append(counts[keep], counts[~keep].sum())
        exp = np.append(expected[keep], expected[~keep].sum())
        if exp[-1] == 0:
            obs, exp = obs[:-1], exp[:-1]
        chi2, pval = stats.chisquare(obs, exp)
        assert pval > 1e-4, (i, chi2, pval)


def test_inputs_are_seeded_and_offsets_differ():
    w = W[1].scaled(B=4, V=256)
    a, b = workloads.make_inputs(w), workloads.make_inputs(w)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    c = workloads.make_inputs(w, seed_offset=1)
    assert not torch.equal(a["target_logits"], c["target_logits"])
    assert not torch.equal(a["u_accept"], c["u_accept"])
    u = torch.cat([a["u_accept"].ravel(), a["u_resample"]])
    assert (u >= 0).all() and (u < 1).all()


@pytest.mark.parametrize("kind", ["chain", "kary:2", "kary:3", "star", "random:3"])
def test_tree_shapes(kind):
    N = 13
    par = workloads.tree_shape(kind, N, seed=4)
    assert len(par) == N + 1 and par[0] == -1
    assert all(0 <= par[j] < j for j in range(1, N + 1))  # parents before children
    name = kind.split(":")[0]
    if name == "chain":
        assert par[1:] == list(range(N))
    elif name == "star":
        assert par[1:] == [0] * N
    elif name == "kary":
        k = int(kind.split(":")[1])
        for u in range(N + 1):
            kids = [j for j in range(1, N + 1) if par[j] == u]
            if kids:  # at most k children, numbered contiguously
                assert len(kids) <= k and kids == list(range(kids[0], kids[0] + len(kids)))
    else:
        assert all(j - par[j] <= 3 for j in range(1, N + 1))


def test_tree_inputs_draw_children_from_their_parents_draft_row():
    """Draft rows are numbered in node order over the nodes with children;
    every child's token is a draw from its parent's draft row (its average log
    probability there beats every other draft row of the tree by a wide margin,
    and the token counts pass a chi-square test against that row's softmax)."""
    from scipy import stats
    B, N, V = 3000, 6, 12
    x = workloads.make_tree_inputs(B, N, V, "f32", "kary:2", s=1.5, a=0.3, e=1.5, seed=3)
    par = x["parent"][0].tolist()
    drow = x["draft_row"][0].tolist()
    assert drow == [0, 1, 2, -1, -1, -1, -1]
    assert (x["parent"] == x["parent"][:1]).all() and (x["draft_row"] == x["draft_row"][:1]).all()
    zq = _np(x["draft_logits"])                        # [B][M][V]
    logq = zq - zq.max(-1, keepdims=True)
    logq -= np.log(np.exp(logq).sum(-1, keepdims=True))
    tok = x["tokens"].numpy()
    M = zq.shape[1]
    for j in range(1, N + 1):
        own = drow[par[j]]
        ll = [float(np.mean(logq[np.arange(B), r, tok[:, j]])) for r in range(M)]
        assert all(ll[own] > ll[r] + 0.1 for r in range(M) if r != own), (j, ll)
        p = np.exp(logq[:, own, :])                    # [B][V]
        counts = np.bincount(tok[:, j], minlength=V)
        chi2, pval = stats.chisquare(counts, p.sum(0))
        assert pval > 1e-4, (j, chi2, pval)
