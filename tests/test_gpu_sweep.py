"""GPU parity of the sweep row kernel (persistent CTAs, chunks staged by bulk
copies) against the fp64 oracle, through the C ABI.

The kernel is forced with SPECV_ROWS_VARIANT=sweep; it takes rows that start
on 16-byte boundaries.  The shapes cover every chunk size the planner picks
(256, 512 and 1024 groups), a row of one short chunk, rows with a ragged last
chunk, rows of many chunks, sampler segments of several tiles, drafts longer
than a warp, and the bonus, residual, invalid and degenerate paths.
"""
import os

import pytest
import torch

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
def sweep_env():
    old = os.environ.get("SPECV_ROWS_VARIANT")
    os.environ["SPECV_ROWS_VARIANT"] = "sweep"
    yield
    if old is None:
        os.environ.pop("SPECV_ROWS_VARIANT", None)
    else:
        os.environ["SPECV_ROWS_VARIANT"] = old


def _args(x):
    return (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])


def _check(specv, w, x, mode, debug=True):
    plan = specv.plan(w.B, w.K, w.V, 1 if w.dtype == "bf16" else 0, mode)
    assert plan["kernel"] == "rows-sweep", plan
    tok, n = specv.verify(*_args(x), mode=mode)
    dbg = specv.verify_debug(*_args(x), mode=mode) if debug else None
    torch.cuda.synchronize()
    if dbg is not None:
        assert torch.equal(dbg["tokens"], tok) and torch.equal(dbg["n_accepted"], n)
    tok, n = tok.cpu().numpy(), n.cpu().numpy()
    xh = _parity.to_host(x)
    orc = _parity.run_oracle(xh, mode)
    rep = _parity.compare(xh, mode, tok, n, orc)
    if dbg is not None:
        rep.update(_parity.check_probabilities(xh, mode, dbg, orc))
    return rep, tok, n, plan


SHAPES = [
    # (B, K, V, dtype, structure)
    (256, 8, 4096, "f32", "half_equal:3.0:0.85:1.0"),   # many items: 1024-group chunks
    (16, 8, 128256, "f32", "half_equal:3.0:0.85:1.0"),  # the batched shape, 32 chunks a row
    (32, 5, 152064, "bf16", "rho:3.0:0.5:0.95"),        # qwen-shaped
    (1, 8, 128256, "bf16", "corr:3.0:0.9:0.7"),         # one sequence: 256-group chunks
    (4, 4, 128256, "bf16", "corr:3.0:0.9:0.7"),         # 512-group chunks
    (1, 4, 1000, "f32", "corr:2.0:0.8:1.0"),            # a row of one short chunk
    (3, 1, 20004, "f32", "corr:2.0:0.8:1.0"),           # K = 1, ragged last chunk
    (2, 40, 4104, "bf16", "rho:3.0:0.5:0.95"),          # K past one warp of positions
    (4, 3, 300000, "f32", "half_equal:3.0:0.85:1.0"),   # sampler segments of two tiles
    (5, 2, 264, "bf16", "corr:3.0:0.9:0.7"),            # V just past the tile kernels
]


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}")
def test_sweep_parity(specv, sweep_env, shape, mode):
    B, K, V, dt, st = shape
    w = workloads.Workload("sweep", B, K, V, dt, st, (0.3,), 13)
    x = workloads.make_inputs(w, DEV)
    rep, _, n, plan = _check(specv, w, x, mode)
    print(f"{shape} mode={mode} plan={plan}: {rep}")


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("cfg", [2, 3])
def test_sweep_on_workloads(specv, sweep_env, cfg, mode):
    w = workloads.WORKLOADS[cfg]
    x = workloads.make_inputs(w, DEV)
    rep, _, _, _ = _check(specv, w, x, mode)
    print(f"workload {cfg} mode={mode}: {rep}")


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
def test_sweep_full_size_batched_sampled(specv, sweep_env, mode):
    """B=256, K=8, V=128256 fp32: every sequence's decisions against the oracle
    on a sample of sequences (both halves of the structure)."""
    w = workloads.WORKLOADS[4]
    x = workloads.make_inputs(w, DEV)
    assert specv.plan(w.B, w.K, w.V, 0, mode)["kernel"] == "rows-sweep"
    tok, n = specv.verify(*_args(x), mode=mode)
    torch.cuda.synchronize()
    tok, n = tok.cpu().numpy(), n.cpu().numpy()
    seqs = list(range(0, 8)) + list(range(128, 136)) + [77, 200, 255]
    xh = _parity.to_host(x)
    orc = _parity.run_oracle(xh, mode, seqs)
    rep = _parity.compare(xh, mode, tok, n, orc, seqs)
    assert (n[128:] == w.K).all()  # the second half drafts with the target itself
    assert ((tok[128:, :w.K] == x["draft_tokens"][128:].cpu().numpy())).all()
    assert ((tok[128:, w.K] >= 0) & (tok[128:, w.K] < w.V)).all()
    print(f"full size sampled mode={mode}: {rep}")


def test_sweep_identical_draft_and_degenerate(specv, sweep_env):
    w = workloads.WORKLOADS[4].scaled(B=6, V=8192)
    x = workloads.make_inputs(w, DEV)
    x["draft_logits"] = x["target_logits"][:, :w.K].contiguous()
    for mode in (0, 1):
        for lam in (0.0, 0.2, 1.0):
            x["lam"] = torch.full((w.B,), lam, dtype=torch.float32, device=DEV)
            tok, n = specv.verify(*_args(x), mode=mode)
            torch.cuda.synchronize()
            assert (n.cpu() == w.K).all(), (mode, lam)
            assert torch.equal(tok[:, :w.K], x["draft_tokens"])
    w = workloads.WORKLOADS[3].scaled(B=4, V=5008)
    x = workloads.make_inputs(w, DEV, lam=1.0)
    _, n = specv.verify(*_args(x), mode=0)
    assert (n.cpu() == w.K).all()
    x = workloads.make_inputs(w, DEV)
    x["u_accept"].zero_()
    for mode in (0, 1):
        _, n = specv.verify(*_args(x), mode=mode)
        assert (n.cpu() == w.K).all()


def test_sweep_invalid_inputs(specv, sweep_env):
    w = workloads.WORKLOADS[1].scaled(B=5, V=4100)
    x = workloads.make_inputs(w, DEV)
    x["draft_tokens"][1, 2] = w.V
    x["draft_tokens"][2, 0] = -3
    x["lam"][3] = 1.5
    x["lam"][4] = float("nan")
    tok, n = specv.verify(*_args(x), mode=0)
    torch.cuda.synchronize()
    tok, n = tok.cpu().numpy(), n.cpu().numpy()
    for b in (1, 2, 3, 4):
        assert n[b] == -1 and (tok[b] == -1).all()
    assert n[0] >= 0
    xh = _parity.to_host(x)
    _parity.compare(xh, 0, tok, n, _parity.run_oracle(xh, 0))


def test_sweep_repeat_calls_and_graph(specv, sweep_env):
    """Counters are left at zero: repeated calls, calls of other shapes in
    between, and graph replays all give the first call's results."""
    w = workloads.WORKLOADS[3].scaled(B=8)
    x = workloads.make_inputs(w, DEV)
    t0, n0 = specv.verify(*_args(x))
    other = workloads.make_inputs(workloads.WORKLOADS[2], DEV)
    for _ in range(3):
        specv.verify(*_args(other))
        t1, n1 = specv.verify(*_args(x))
        torch.cuda.synchronize()
        assert torch.equal(t0, t1) and torch.equal(n0, n1)
    tok = torch.empty_like(t0)
    nn = torch.empty_like(n0)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        specv.verify(*_args(x), out_tokens=tok, out_n_accepted=nn,
                     stream=torch.cuda.current_stream())
    for _ in range(3):
        tok.fill_(-9)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(tok, t0) and torch.equal(nn, n0)
