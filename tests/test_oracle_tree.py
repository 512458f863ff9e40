"""Pins for the oracle's tree verification (the reading in specv_oracle.c:
siblings drawn independently from the draft distribution of their parent,
tested in index order, each rejection replacing p by normalize(max(0, p - q)),
an acceptance moving the walk to that child; the pages' "Tree Speculation"
section of the speculative-decoding explainer and "3. 验证阶段树形attention" of
the EAGLE explainer describe the trees, not this rule).

Pinned by: reduction to the pinned chain loop when every node has one child;
the lossless property (the first emitted token is distributed as p~ at the
root) by exact enumeration of the drafted tokens and a rank-1 lattice over the
uniforms; the same two levels deep (the second token, given the first, is
distributed as p~ at the accepted child; this alone catches a walk that skips
the residual update between siblings below the root); hand-worked cases;
invalid inputs.
"""
import math

import numpy as np
import pytest
import torch

import workloads


def _chain_as_tree(x):
    """The chain inputs of verify() as a tree: node j (1..K) is draft j-1, its
    parent is j-1; node u < K draws its child from draft row u; node K is a leaf."""
    zt = x["target_logits"]
    B, K1, V = zt.shape
    K = K1 - 1
    parent = torch.arange(-1, K, dtype=torch.int32).repeat(B, 1)
    drow = torch.arange(0, K + 1, dtype=torch.int32).repeat(B, 1)
    drow[:, K] = -1
    tok = torch.zeros((B, K + 1), dtype=torch.int32)
    tok[:, 1:] = x["draft_tokens"].cpu()
    ua = torch.zeros((B, K + 1), dtype=torch.float32)
    ua[:, 1:] = x["u_accept"].cpu()
    return parent, drow, tok, ua


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("cfg", [1, 3, 5])
def test_tree_with_one_child_per_node_is_the_chain(oracle_mod, cfg, mode):
    w = workloads.WORKLOADS[cfg].scaled(B=min(workloads.WORKLOADS[cfg].B, 64), V=2003
                                        if cfg == 3 else workloads.WORKLOADS[cfg].V)
    x = workloads.make_inputs(w, "cpu")
    chain = oracle_mod.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                              x["u_accept"], x["u_resample"], x["lam"], mode=mode)
    parent, drow, tok, ua = _chain_as_tree(x)
    tree = oracle_mod.verify_tree(x["target_logits"], x["draft_logits"], parent, drow, tok, ua,
                                  x["u_resample"], x["lam"], mode=mode)
    np.testing.assert_array_equal(tree.n_accepted, chain.n_accepted)
    np.testing.assert_array_equal(tree.tokens, chain.tokens)
    np.testing.assert_allclose(tree.accept_margin, chain.accept_margin, rtol=0, atol=1e-12)
    np.testing.assert_allclose(tree.cdf_margin, chain.cdf_margin, rtol=0, atol=1e-12)
    n = tree.n_accepted
    for b in range(w.B):  # the path is the chain 1..n
        assert tree.path[b, :n[b]].tolist() == list(range(1, n[b] + 1))


def _lattice(n, dims, gen):
    """Rank-1 lattice {frac(k * g / n)} in [0,1)^dims, shifted by half a cell."""
    k = np.arange(n)[:, None]
    return np.mod((k * np.array(gen[:dims])[None, :] + 0.5) / n, 1.0)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("lam", [0.0, 0.4])
@pytest.mark.parametrize("children", [2, 3])
def test_tree_is_lossless_at_the_root(oracle_mod, mode, lam, children):
    """Root with `children` leaves drawn i.i.d. from q: over every draw of the
    children's tokens (weighted by their probability) and a lattice over the
    uniforms, the first emitted token is distributed as p~ at the root."""
    V = 3
    rng = np.random.default_rng(17 + children)
    zt = rng.normal(0, 1.2, (1, children + 1, V)).astype(np.float32)
    zq = rng.normal(0, 1.2, (1, 1, V)).astype(np.float32)
    ptilde, q = oracle_mod.rows(zt[0, :2], zq[0, :1], lam, mode)
    p_root, q_root = ptilde[0], q[0]
    n = 1 << 13
    gens = {2: (1, 1433, 3319), 3: (1, 1433, 3319, 5879)}[children]
    uni = _lattice(n, children + 1, gens + (0,) * 4)
    dist = np.zeros(V)
    parent = np.array([[-1] + [0] * children], np.int32).repeat(n, 0)
    drow = np.array([[0] + [-1] * children], np.int32).repeat(n, 0)
    for combo in np.ndindex(*([V] * children)):
        weight = float(np.prod([q_root[c] for c in combo]))
        tok = np.array([[0] + list(combo)], np.int32).repeat(n, 0)
        ua = np.zeros((n, children + 1), np.float32)
        ua[:, 1:] = uni[:, :children]
        ur = uni[:, children].astype(np.float32)
        r = oracle_mod.verify_tree(np.broadcast_to(zt, (n,) + zt.shape[1:]),
                                   np.broadcast_to(zq, (n,) + zq.shape[1:]), parent, drow, tok,
                                   ua, ur, np.full(n, lam, np.float32), mode=mode)
        first = r.tokens[:, 0]
        dist += weight * np.bincount(first, minlength=V) / n
    np.testing.assert_allclose(dist, p_root, atol=2e-3)


def _softmax64(z):
    e = np.exp(np.asarray(z, np.float64) - np.max(z))
    return e / e.sum()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("lam", [0.0, 0.35])
def test_tree_is_lossless_two_levels_deep(oracle_mod, mode, lam):
    """Root with two children, each with two leaf children (V = 3).  As for a
    real model, a node's target row and the draft row of its children depend
    only on the tokens of its path.  Over every draw of the six drafted tokens
    (weighted by their probability under the drafting node's q) and a scrambled
    Sobol set of the seven uniforms: the first token is distributed as p~ at the
    root and, when a child was accepted (n >= 1), the second token given the
    first token a is distributed as p~ at the child holding a.  A walk that kept
    the root's p after an acceptance, tested the leaves against the root's q or
    drew them from the wrong row would break the second statement."""
    qmc = pytest.importorskip("scipy.stats.qmc")
    V = 3
    rng = np.random.default_rng(29)
    R0 = rng.normal(0, 1.1, V).astype(np.float32)         # root target row
    Q0 = rng.normal(0, 1.1, V).astype(np.float32)         # root's draft row
    R1 = rng.normal(0, 1.1, (V, V)).astype(np.float32)    # target row of a child holding a
    Q1 = rng.normal(0, 1.1, (V, V)).astype(np.float32)    # its draft row
    R2 = rng.normal(0, 1.1, (V, V, V)).astype(np.float32)  # leaf rows (bonus only)
    pad = np.zeros(V, np.float32)
    p_root = oracle_mod.rows(np.stack([R0, pad]), Q0[None], lam, mode)[0][0]
    p_child = np.stack([oracle_mod.rows(np.stack([R1[a], pad]), Q1[a][None], lam, mode)[0][0]
                        for a in range(V)])
    # the second statement can tell the child's p~ from the root's
    assert np.abs(p_child - p_root[None]).max() > 0.1
    q0 = _softmax64(Q0)
    q1 = np.stack([_softmax64(Q1[a]) for a in range(V)])

    n = 1 << 11
    u = qmc.Sobol(d=7, scramble=True, seed=5).random_base2(m=11).astype(np.float32)
    u = np.minimum(u, np.nextafter(np.float32(1), np.float32(0)))
    leaves = np.array(list(np.ndindex(V, V, V, V)), np.int32)  # tokens of nodes 3, 4, 5, 6
    L = len(leaves)
    B = L * n
    parent = np.tile(np.array([-1, 0, 0, 1, 1, 2, 2], np.int32), (B, 1))
    drow = np.tile(np.array([0, 1, 2, -1, -1, -1, -1], np.int32), (B, 1))
    ua = np.zeros((B, 7), np.float32)
    ua[:, 1:] = np.tile(u[:, :6], (L, 1))
    ur = np.tile(u[:, 6], L)
    lam_b = np.full(B, lam, np.float32)
    first = np.zeros(V)
    reached = np.zeros(V)        # P(first token a, a child accepted)
    joint = np.zeros((V, V))     # P(first token a, a child accepted, second token c)
    for t1, t2 in np.ndindex(V, V):
        tok = np.zeros((B, 7), np.int32)
        tok[:, 1], tok[:, 2] = t1, t2
        tok[:, 3:] = np.repeat(leaves, n, axis=0)
        zt = np.empty((B, 7, V), np.float32)
        zt[:, 0], zt[:, 1], zt[:, 2] = R0, R1[t1], R1[t2]
        for j, par_tok in ((3, t1), (4, t1), (5, t2), (6, t2)):
            zt[:, j] = R2[par_tok][tok[:, j]]
        zq = np.empty((B, 3, V), np.float32)
        zq[:, 0], zq[:, 1], zq[:, 2] = Q0, Q1[t1], Q1[t2]
        r = oracle_mod.verify_tree(zt, zq, parent, drow, tok, ua, ur, lam_b, mode=mode)
        w = q0[t1] * q0[t2] * np.prod(
            [q1[t1][leaves[:, 0]], q1[t1][leaves[:, 1]], q1[t2][leaves[:, 2]],
             q1[t2][leaves[:, 3]]], axis=0)                 # [L]
        wb = np.repeat(w, n) / n                            # weight of each sequence
        t0, s1 = r.tokens[:, 0], r.tokens[:, 1]
        acc = r.n_accepted >= 1
        for a in range(V):
            first[a] += wb[t0 == a].sum()
            reached[a] += wb[(t0 == a) & acc].sum()
            for c in range(V):
                joint[a, c] += wb[(t0 == a) & acc & (s1 == c)].sum()
    assert abs(first.sum() - 1.0) < 1e-9
    np.testing.assert_allclose(first, p_root, atol=4e-3)
    assert reached.min() > 0.05
    np.testing.assert_allclose(joint, reached[:, None] * p_child, atol=4e-3)


def test_tree_hand_cases(oracle_mod):
    # p~ at the root = (0.8, 0.2) (lambda = 0, probability mode), q = (0.5, 0.5).
    zt = np.log(np.array([[[0.8, 0.2], [0.1, 0.9], [0.6, 0.4]]])).astype(np.float32)
    zq = np.log(np.array([[[0.5, 0.5]]])).astype(np.float32)
    parent = np.array([[-1, 0, 0]], np.int32)
    drow = np.array([[0, -1, -1]], np.int32)
    lam = np.array([0.0], np.float32)
    # both children draft token 1: ratio 0.2/0.5 = 0.4 -> u = 0.5 rejects; the
    # residual is (0.3, 0)/0.3 = (1, 0), so the second token 1 has ratio 0 and
    # is rejected too; the residual of (1, 0) - (0.5, 0.5) is (1, 0): token 0.
    r = oracle_mod.verify_tree(zt, zq, parent, drow, np.array([[0, 1, 1]], np.int32),
                               np.array([[0, 0.5, 0.0]], np.float32),
                               np.array([0.7], np.float32), lam)
    assert r.n_accepted.tolist() == [0] and r.tokens.tolist() == [[0, -1, -1]]
    # first child (token 1) rejected at u = 0.5; second child token 0: under the
    # residual (1, 0) its ratio is 1 / 0.5 = 2 -> accepted; node 2 is a leaf:
    # bonus from its target row (0.6, 0.4) at u = 0.7 -> token 1.
    r = oracle_mod.verify_tree(zt, zq, parent, drow, np.array([[0, 1, 0]], np.int32),
                               np.array([[0, 0.5, 0.99]], np.float32),
                               np.array([0.7], np.float32), lam)
    assert r.n_accepted.tolist() == [1]
    assert r.path.tolist() == [[2, -1, -1]] and r.tokens.tolist() == [[0, 1, -1]]
    # first child accepted (u = 0.3 < 0.4): walk to node 1 (leaf, row (0.1, 0.9));
    # bonus at u = 0.05 -> token 0
    r = oracle_mod.verify_tree(zt, zq, parent, drow, np.array([[0, 1, 0]], np.int32),
                               np.array([[0, 0.3, 0.0]], np.float32),
                               np.array([0.05], np.float32), lam)
    assert r.path.tolist() == [[1, -1, -1]] and r.tokens.tolist() == [[1, 0, -1]]


@pytest.mark.parametrize("breakage", ["root_parent", "forward_parent", "no_draft_row",
                                      "draft_row_range", "token", "lambda"])
def test_tree_invalid_inputs(oracle_mod, breakage):
    V, N, M = 5, 3, 2
    zt = np.zeros((2, N + 1, V), np.float32)
    zq = np.zeros((2, M, V), np.float32)
    parent = np.array([[-1, 0, 0, 1]] * 2, np.int32)
    drow = np.array([[0, 1, -1, -1]] * 2, np.int32)
    tok = np.array([[0, 1, 2, 3]] * 2, np.int32)
    lam = np.array([0.3, 0.3], np.float32)
    if breakage == "root_parent":
        parent[1, 0] = 0
    elif breakage == "forward_parent":
        parent[1, 2] = 2
    elif breakage == "no_draft_row":
        drow[1, 1] = -1  # node 1 has a child (node 3)
    elif breakage == "draft_row_range":
        drow[1, 2] = M
    elif breakage == "token":
        tok[1, 3] = V
    else:
        lam[1] = -0.5
    r = oracle_mod.verify_tree(zt, zq, parent, drow, tok, np.zeros((2, N + 1), np.float32),
                               np.zeros(2, np.float32), lam)
    assert r.n_accepted[1] == -1 and (r.tokens[1] == -1).all() and (r.path[1] == -1).all()
    assert r.n_accepted[0] >= 0
