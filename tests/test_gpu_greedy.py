"""GPU parity of greedy verification (mode GREEDY) against the fp64 oracle.

The kernels form the mixed logit w = z_t + lambda (z_q - z_t) in fp32, the
oracle (1 - lambda) z_t + lambda z_q in double precision.  Every sequence
whose decided rows are farther from a tie than the band derived in
tests/_parity.py (GREEDY_BAND, relative to the row's largest |logit|) must
match bit for bit: n_accepted and every emitted token.  Near-ties are counted
and the GPU's output there must be a valid greedy outcome (accepted drafts and
the emitted token near-maxima of their rows, the bonus the exact argmax of
target row K).  Exact ties go to the smallest index; inputs with many equal
logits check that rule across threads, warps, CTAs and cluster ranks.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def specv():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    import speculative_decoding_verification_specv_gb300 as m
    m.load(build_if_missing=True)
    return m


@pytest.fixture
def env_guard():
    keys = ("SPECV_CLUSTER_SIZE", "SPECV_ROWS_VARIANT")
    old = {k: os.environ.get(k) for k in keys}
    yield
    for k, v in old.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def _follow_argmax(x, frac=0.5, seed=0):
    """Replace the draft tokens of a fraction of the sequences by the greedy
    argmax of every drafted row (computed by the oracle), so that long
    accepted prefixes and the bonus path are exercised."""
    rng = np.random.default_rng(seed)
    zt = x["target_logits"].float().cpu().numpy()
    zq = x["draft_logits"].float().cpu().numpy()
    lam = x["lam"].cpu().numpy()
    tok = x["draft_tokens"].cpu().numpy().copy()
    B, K = tok.shape
    for b in range(B):
        if rng.random() < frac:
            # follow all rows, or stop following at a random position
            stop = K if rng.random() < 0.5 else int(rng.integers(0, K))
            for i in range(stop):
                tok[b, i] = oracle.greedy_argmax(zt[b, i], zq[b, i], lam[b])
    x["draft_tokens"] = torch.from_numpy(tok).to(DEV)
    return x


def _check(specv, x, seqs=None):
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    tok, n = specv.verify(*args, mode=specv.GREEDY)
    torch.cuda.synchronize()
    tok, n = tok.cpu().numpy(), n.cpu().numpy()
    xh = _parity.to_host(x)
    if seqs is None:
        orc = oracle.verify_greedy(xh["target_logits"], xh["draft_logits"], xh["draft_tokens"],
                                   xh["lam"])
    else:
        idx = torch.as_tensor(seqs)
        sub = {k: v.index_select(0, idx) for k, v in xh.items()}
        orc = oracle.verify_greedy(sub["target_logits"], sub["draft_logits"],
                                   sub["draft_tokens"], sub["lam"])
    rep = _parity.compare_greedy(xh, tok, n, orc, seqs=seqs)
    print("greedy parity:", rep)
    return tok, n


SMALL = {
    1: workloads.WORKLOADS[1],
    2: workloads.WORKLOADS[2],
    3: workloads.WORKLOADS[3],
    4: workloads.WORKLOADS[4].scaled(B=16),
    5: workloads.WORKLOADS[5].scaled(B=20_000),
}


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_greedy_workloads(specv, cfg):
    w = SMALL[cfg]
    x = _follow_argmax(workloads.make_inputs(w, DEV), seed=cfg)
    tok, n = _check(specv, x)
    plan = specv.plan(w.B, w.K, w.V, 1 if w.dtype == "bf16" else 0, 2)
    print(f"greedy workload {cfg}: plan={plan} mean n={n.mean():.3f} "
          f"all-accepted={(n == w.K).mean():.3f}")


def test_greedy_full_size_batched_sampled(specv):
    w = workloads.WORKLOADS[4]
    x = _follow_argmax(workloads.make_inputs(w, DEV), frac=0.5, seed=4)
    seqs = list(range(0, 256, 9)) + [255]
    _check(specv, x, seqs)


def test_greedy_full_size_exactness_workload(specv):
    w = workloads.WORKLOADS[5]
    x = workloads.make_inputs(w, DEV)
    # 2% of the 10^6 sequences draft the greedy argmax (long prefixes, bonus
    # path); the rest draft sampled tokens
    x = _follow_argmax(x, frac=0.02, seed=5)
    _check(specv, x)


@pytest.mark.parametrize("lam", [0.0, 0.3, 1.0])
@pytest.mark.parametrize("shape", [(3, 1, 1001, "f32"), (5, 3, 33, "f32"), (2, 4, 515, "bf16"),
                                   (7, 2, 256, "bf16"), (41, 4, 32, "f32"), (1, 1, 1, "f32"),
                                   (2, 40, 4104, "bf16"), (2, 3, 131071, "f32")],
                         ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}" if isinstance(s, tuple) else s)
def test_greedy_ragged_shapes(specv, shape, lam):
    B, K, V, dt = shape
    w = workloads.Workload("ragged", B, K, V, dt, "corr:2.0:0.8:1.0", (lam,), 21)
    x = _follow_argmax(workloads.make_inputs(w, DEV), frac=0.7, seed=V)
    _check(specv, x)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 7, 8, 16])
def test_greedy_every_cluster_size_with_ties(specv, env_guard, S):
    """Integer logits in a small range: every row has many equal maxima, spread
    over all ranks of the cluster; the first one in index order must win."""
    os.environ["SPECV_CLUSTER_SIZE"] = str(S)
    B, K, V = 6, 3, 50000
    g = torch.Generator().manual_seed(100 + S)
    zt = torch.randint(-3, 4, (B, K + 1, V), generator=g).float()
    zq = torch.randint(-3, 4, (B, K, V), generator=g).float()
    x = {"target_logits": zt.to(DEV), "draft_logits": zq.to(DEV),
         "draft_tokens": torch.zeros((B, K), dtype=torch.int32, device=DEV),
         "u_accept": torch.rand((B, K), generator=g).to(DEV),
         "u_resample": torch.rand((B,), generator=g).to(DEV),
         "lam": torch.tensor([0.0, 0.5, 0.25, 1.0, 0.0, 0.75], dtype=torch.float32, device=DEV)}
    p = specv.plan(B, K, V, 0, 2)
    assert p["cluster"] == S and p["kernel"] == "rows-stream"
    x = _follow_argmax(x, frac=0.6, seed=S)
    _check(specv, x)
    # the all-equal row: the argmax is index 0
    x["target_logits"][0].fill_(2.0)
    x["draft_logits"][0].fill_(2.0)
    tok, n = _check(specv, x)
    assert tok[0, n[0]] == 0


def test_greedy_masked_draft_entries_and_invalid_inputs(specv):
    w = workloads.WORKLOADS[3].scaled(B=6)
    x = workloads.make_inputs(w, DEV)
    # the target's best entries are ruled out by -inf draft logits
    best = x["target_logits"][:, :w.K].argmax(-1)
    x["draft_logits"].scatter_(-1, best.unsqueeze(-1), float("-inf"))
    x["draft_tokens"][1, 2] = w.V
    x["draft_tokens"][2, 0] = -3
    x["lam"][3] = 1.5
    x["lam"][4] = float("nan")
    tok, n = _check(specv, x)
    for b in (1, 2, 3, 4):
        assert n[b] == -1 and (tok[b] == -1).all()


def test_greedy_noalloc_and_debug(specv):
    w = workloads.WORKLOADS[3].scaled(B=4)
    x = _follow_argmax(workloads.make_inputs(w, DEV), frac=0.5, seed=8)
    ref_tok, ref_n = _check(specv, x)
    tok = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=DEV)
    n = torch.empty((w.B,), dtype=torch.int32, device=DEV)
    fn = specv.load().specv_verify_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_int, ctypes.c_int, vp, vp, vp]
    fn.restype = ctypes.c_int
    st = fn(x["target_logits"].data_ptr(), x["draft_logits"].data_ptr(),
            x["draft_tokens"].data_ptr(), x["u_accept"].data_ptr(), x["u_resample"].data_ptr(),
            x["lam"].data_ptr(), w.B, w.K, w.V, 1, 2, tok.data_ptr(), n.data_ptr(),
            vp(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok)
    np.testing.assert_array_equal(n.cpu().numpy(), ref_n)
    with pytest.raises(specv.SpecvError):
        specv.verify_debug(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                           x["u_accept"], x["u_resample"], x["lam"], mode=specv.GREEDY)
