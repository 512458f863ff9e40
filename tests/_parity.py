"""Comparison of the CUDA verify step with the fp64 oracle (test helper).

Decisions are compared exactly except where a uniform lies within BAND of a
decision boundary: |u_i - min(1, ratio_i)| for a decided position, or the
distance of u_resample to the nearest boundary of the CDF it was drawn
through.  Those sequences are counted, and their GPU output must still be a
valid outcome: an accepted prefix of the draft, then one token that has
positive probability under the distribution of that step, then -1; when the
GPU took the oracle's acceptance decisions, that token must also lie in the
oracle's inverse-CDF interval of u_resample to within the band.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

BAND = 1e-5          # decision-boundary band
# Greedy tie band, relative to the row's largest |logit| A.  The kernels form
# w = z_t + lam (z_q - z_t) in fp32 (one rounded subtraction, one fused
# multiply-add): |w32 - w| <= u (lam |z_q - z_t| + |w|)(1 + u) <= 3 u A (1 + u)
# with u = 2^-24, so two entries whose exact scores differ by more than
# 6 u A (1 + u) < 2^-21 A are ordered the same way in fp32 as in fp64.  Rows
# whose fp64 gap between the best and the second-best score is below
# 2^-20 A (a factor 2 of margin) count as near-ties.
GREEDY_BAND = 2.0 ** -20
TOL_F32 = 1e-5       # |p_gpu - p_oracle| for fp32 logits
TOL_BF16 = 2e-3      # |p_gpu - p_oracle| for bf16 logits


def to_host(x):
    return {k: (v.detach().cpu() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def run_oracle(xh, mode, seqs=None):
    """Oracle on all sequences, or on the listed ones (a gathered sub-batch)."""
    if seqs is not None:
        idx = torch.as_tensor(seqs, dtype=torch.long)
        xh = {k: v.index_select(0, idx) for k, v in xh.items()}
    return oracle.verify(xh["target_logits"], xh["draft_logits"], xh["draft_tokens"],
                         xh["u_accept"], xh["u_resample"], xh["lam"], mode=mode)


def _valid_outcome(xh_b, mode, n, toks, same_n=False, band=BAND):
    """Is (n, toks) a possible output for this sequence?  With same_n (the GPU
    took the oracle's decisions), the drawn token must also lie in the oracle's
    fp64 inverse-CDF interval of u_resample for that step's distribution, to
    within the band: C_{t-1} - band <= u <= C_t + band."""
    K = xh_b["draft_tokens"].shape[0]
    if not (0 <= n <= K):
        return False
    drafts = xh_b["draft_tokens"].numpy()
    if list(toks[:n]) != list(drafts[:n]) or any(t != -1 for t in toks[n + 1:]):
        return False
    t = int(toks[n])
    V = xh_b["target_logits"].shape[-1]
    if not (0 <= t < V):
        return False
    lam = float(xh_b["lam"])
    pt, q = oracle.rows(xh_b["target_logits"], xh_b["draft_logits"], lam, mode)
    if n == K:
        w = pt[K]
    else:
        w = np.maximum(0.0, pt[n] - q[n])
        if w.sum() < 1e-12:
            w = pt[n]
    if not w[t] > 0:
        return False
    if not same_n:
        return True
    c = np.cumsum(w) / w.sum()
    lo = c[t - 1] if t > 0 else 0.0
    u = float(xh_b["u_resample"])
    return lo - band <= u <= c[t] + band


def compare(xh, mode, gpu_tokens, gpu_n, orc, seqs=None, band=BAND):
    """Returns a report dict; raises AssertionError on any mismatch outside the band."""
    gt = np.asarray(gpu_tokens)
    gn = np.asarray(gpu_n)
    seqs = list(range(gn.shape[0])) if seqs is None else list(seqs)
    near = exact = near_same = 0
    mism = []
    near_tight = 0
    for j, b in enumerate(seqs):
        on, ot = int(orc.n_accepted[j]), orc.tokens[j]
        if on == -1:
            if not (gn[b] == -1 and (gt[b] == -1).all()):
                mism.append((b, "invalid", on, gn[b]))
            continue
        am, cm = float(orc.accept_margin[j]), float(orc.cdf_margin[j])
        if am < band or cm < band:
            near += 1
            if am < 1e-7 or cm < 1e-7:
                near_tight += 1
            if gn[b] == on and (gt[b] == ot).all():
                near_same += 1
                continue
            xb = {k: v[b] for k, v in xh.items()}
            if not _valid_outcome(xb, mode, int(gn[b]), gt[b], same_n=int(gn[b]) == on):
                mism.append((b, "invalid-outcome-near-band", on, int(gn[b]), ot.tolist(),
                             gt[b].tolist()))
            continue
        if gn[b] != on or not (gt[b] == ot).all():
            mism.append((b, "mismatch", on, int(gn[b]), ot.tolist(), gt[b].tolist(), am, cm))
        else:
            exact += 1
    rep = dict(sequences=len(seqs), exact=exact, near_band=near, near_band_same=near_same,
               near_band_1e7=near_tight, mismatches=len(mism))
    assert not mism, f"{len(mism)} mismatches outside the {band} band: {mism[:5]} report={rep}"
    return rep


def check_probabilities(xh, mode, dbg, orc, seqs=None):
    """p~(x_i), q(x_i) against the oracle within the dtype's tolerance."""
    tol = TOL_BF16 if xh["target_logits"].dtype == torch.bfloat16 else TOL_F32
    seqs = list(range(dbg["ptilde_x"].shape[0])) if seqs is None else list(seqs)
    px = dbg["ptilde_x"].cpu().numpy()[seqs]
    qx = dbg["q_x"].cpu().numpy()[seqs]
    ok = ~np.isnan(orc.ptilde_x)
    err_p = np.abs(px - orc.ptilde_x)[ok].max(initial=0.0)
    err_q = np.abs(qx - orc.q_x)[ok].max(initial=0.0)
    rel_p = (np.abs(px - orc.ptilde_x) / np.maximum(orc.ptilde_x, 1e-30))[ok].max(initial=0.0)
    assert err_p <= tol and err_q <= tol, (err_p, err_q, tol)
    return dict(max_abs_err_ptilde=float(err_p), max_abs_err_q=float(err_q),
                max_rel_err_ptilde=float(rel_p))


def check_rows(xh, mode, dbg, seqs, tol=None):
    """Whole rows: the distributions implied by the GPU's log-normalisers
    (p_t,v = exp(z_t,v - lse_A), q_v = exp(z_q,v - lse_B); in logit mode the
    A row is the mixed row, formed in fp32 as the kernels form it) against the
    oracle's fp64 p~ and q rows, entry by entry, for the listed sequences."""
    if tol is None:
        tol = TOL_BF16 if xh["target_logits"].dtype == torch.bfloat16 else TOL_F32
    lse = dbg["lse"].cpu().numpy().astype(np.float64)
    worst_p = worst_q = 0.0
    for b in seqs:
        zt32 = xh["target_logits"][b].float().numpy()
        zq32 = xh["draft_logits"][b].float().numpy()
        lam = float(xh["lam"][b])
        pt_o, q_o = oracle.rows(xh["target_logits"][b], xh["draft_logits"][b], lam, mode)
        K = zq32.shape[0]
        for j in range(K + 1):
            if j < K:
                qg = np.exp(zq32[j].astype(np.float64) - lse[b, j, 1])
                if mode == oracle.PROB_MIX:
                    ptg = np.exp(zt32[j].astype(np.float64) - lse[b, j, 0])
                    pg = (1.0 - lam) * ptg + lam * qg
                else:
                    lam32 = np.float32(lam)
                    if lam32 == 0 or lam32 == 1:  # a zero-weight term drops out exactly
                        w = zt32[j] if lam32 == 0 else zq32[j]
                    else:
                        with np.errstate(invalid="ignore"):
                            w = (zt32[j] + lam32 * (zq32[j] - zt32[j])).astype(np.float32)
                        w = np.where(np.isnan(w), -np.inf, w)  # a masked entry of weight > 0
                    pg = np.exp(w.astype(np.float64) - lse[b, j, 0])
                worst_q = max(worst_q, float(np.abs(qg - q_o[j]).max()))
            else:  # the bonus row: the target softmax
                pg = np.exp(zt32[j].astype(np.float64) - lse[b, j, 0])
            worst_p = max(worst_p, float(np.abs(pg - pt_o[j]).max()))
    assert worst_p <= tol and worst_q <= tol, (worst_p, worst_q, tol)
    return dict(max_abs_err_ptilde_rows=worst_p, max_abs_err_q_rows=worst_q)


def _near_argmax(w, A, t, band):
    return np.isfinite(w[t]) and w[t] >= w.max() - band * A or w[t] == w.max()


def _valid_greedy_outcome(xh_b, n, toks, band=GREEDY_BAND):
    """Is (n, toks) a greedy outcome that fp32 rounding of the scores could
    give?  Every accepted draft is a near-maximum of its row, the token at a
    mismatch is a near-maximum of that row other than the draft, and a bonus
    token is the exact argmax of target row K (w = z_t there, no rounding)."""
    K = xh_b["draft_tokens"].shape[0]
    if not (0 <= n <= K):
        return False
    drafts = xh_b["draft_tokens"].numpy()
    if list(toks[:n]) != list(drafts[:n]) or any(t != -1 for t in toks[n + 1:]):
        return False
    zt = xh_b["target_logits"].float().numpy()
    zq = xh_b["draft_logits"].float().numpy()
    lam = float(xh_b["lam"])
    V = zt.shape[-1]

    def row(i):
        w = oracle.greedy_scores(zt[i], zq[i], lam)
        a = np.abs(np.concatenate([zt[i], zq[i]]).astype(np.float64))
        A = float(a[np.isfinite(a)].max(initial=0.0))
        return w, A
    for i in range(n):
        w, A = row(i)
        if not _near_argmax(w, A, int(drafts[i]), band):
            return False
    t = int(toks[n])
    if not (0 <= t < V):
        return False
    if n == K:
        return t == oracle.greedy_argmax(zt[K], None, lam)
    w, A = row(n)
    return t != int(drafts[n]) and _near_argmax(w, A, t, band)


def compare_greedy(xh, gpu_tokens, gpu_n, orc, seqs=None, band=GREEDY_BAND):
    """Greedy outputs against the fp64 oracle: bit-exact for every sequence
    whose decided rows are all farther than the band from a tie; within the
    band, counted, and the GPU's output must be a valid greedy outcome.
    Raises AssertionError on any mismatch outside the band."""
    gt = np.asarray(gpu_tokens)
    gn = np.asarray(gpu_n)
    seqs = list(range(gn.shape[0])) if seqs is None else list(seqs)
    near = exact = near_same = 0
    mism = []
    for j, b in enumerate(seqs):
        on, ot = int(orc.n_accepted[j]), orc.tokens[j]
        if on == -1:
            if not (gn[b] == -1 and (gt[b] == -1).all()):
                mism.append((b, "invalid", on, int(gn[b])))
            continue
        same = gn[b] == on and (gt[b] == ot).all()
        if float(orc.tie_margin[j]) < band:
            near += 1
            if same:
                near_same += 1
                continue
            xb = {k: v[b] for k, v in xh.items()}
            if not _valid_greedy_outcome(xb, int(gn[b]), gt[b], band):
                mism.append((b, "invalid-outcome-near-tie", on, int(gn[b]), ot.tolist(),
                             gt[b].tolist()))
            continue
        if not same:
            mism.append((b, "mismatch", on, int(gn[b]), ot.tolist(), gt[b].tolist(),
                         float(orc.tie_margin[j])))
        else:
            exact += 1
    rep = dict(sequences=len(seqs), exact=exact, near_tie=near, near_tie_same=near_same,
               mismatches=len(mism))
    assert not mism, f"{len(mism)} greedy mismatches outside the tie band: {mism[:5]} report={rep}"
    return rep


def compare_tree(xh, gpu_tokens, gpu_path, gpu_n, orc, band=BAND):
    """Tree verification against the oracle: exact (n, tokens, path) outside
    the decision band; inside it the GPU's walk must still be valid (each
    accepted node a child of the previous one, carrying its token, then one
    token in [0, V), then -1).  Returns (exact, near)."""
    tok, path, n = (np.asarray(a) for a in (gpu_tokens, gpu_path, gpu_n))
    par = np.asarray(xh["parent"])
    ntok = np.asarray(xh["tokens"])
    V = xh["target_logits"].shape[-1]
    exact = near = 0
    for b in range(n.shape[0]):
        on = int(orc.n_accepted[b])
        if on == -1:
            assert n[b] == -1 and (tok[b] == -1).all() and (path[b] == -1).all(), b
            continue
        if orc.accept_margin[b] >= band and orc.cdf_margin[b] >= band:
            assert n[b] == on, (b, n[b], on)
            np.testing.assert_array_equal(tok[b], orc.tokens[b])
            np.testing.assert_array_equal(path[b], orc.path[b])
            exact += 1
            continue
        near += 1
        k = int(n[b])
        assert 0 <= k <= par.shape[1] - 1
        prev = 0
        for j in range(k):
            c = int(path[b, j])
            assert par[b, c] == prev and tok[b, j] == ntok[b, c]
            prev = c
        assert 0 <= tok[b, k] < V
        assert (tok[b, k + 1:] == -1).all() and (path[b, k:] == -1).all()
    return exact, near
