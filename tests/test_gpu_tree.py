"""GPU parity of tree verification (specv_verify_tree) against the oracle.

Decisions must match the oracle exactly (n, every emitted token, the accepted
path) except in sequences where a uniform lies within 1e-5 of a decision or
CDF boundary; those are counted and must still hold a valid walk (each accepted
node a child of the previous one, its token the node's token, the drawn token
inside the vocabulary, -1 after).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BAND = 1e-5


@pytest.fixture(scope="module")
def specv():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    import speculative_decoding_verification_specv_gb300 as m
    m.load(build_if_missing=True)
    return m


@pytest.fixture
def env_guard():
    old = os.environ.get("SPECV_CLUSTER_SIZE")
    yield
    if old is None:
        os.environ.pop("SPECV_CLUSTER_SIZE", None)
    else:
        os.environ["SPECV_CLUSTER_SIZE"] = old


def _args(x):
    return (x["target_logits"], x["draft_logits"], x["parent"], x["draft_row"], x["tokens"],
            x["u_accept"], x["u_resample"], x["lam"])


def _check(specv, x, mode):
    tok, path, n = specv.verify_tree(*_args(x), mode=mode)
    torch.cuda.synchronize()
    tok, path, n = tok.cpu().numpy(), path.cpu().numpy(), n.cpu().numpy()
    orc = oracle.verify_tree(*[v.cpu() for v in _args(x)], mode=mode)
    _, near = _parity.compare_tree({k: v.cpu() for k, v in x.items()}, tok, path, n, orc)
    return n, near


SHAPES = [
    # (B, N, V, dtype, tree)
    (16, 12, 4099, "f32", "kary:2"),
    (16, 12, 4104, "bf16", "kary:3"),
    (8, 20, 2048, "f32", "random:4"),
    (6, 9, 33, "f32", "star"),
    (4, 15, 128256, "bf16", "kary:2"),
    (32, 6, 1000, "f32", "chain"),
    (5, 0, 777, "f32", "chain"),          # root only: the bonus draw
    (3, 40, 513, "bf16", "random:8"),
]


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}N{s[1]}V{s[2]}{s[3]}-{s[4]}")
def test_tree_parity(specv, shape, mode):
    B, N, V, dt, tree = shape
    for lam, seed in ((0.0, 1), (0.3, 2)):
        x = workloads.make_tree_inputs(B, N, V, dt, tree, lam=lam, seed=seed, device=DEV)
        n, near = _check(specv, x, mode)
        print(f"{shape} mode={mode} lam={lam}: mean n={n.mean():.2f}, near-boundary={near}")


def test_tree_many_siblings_rejected(specv):
    """A star of 24 children drawn from a draft that disagrees with the target:
    most children are rejected, each rejection a pass over the root's rows."""
    x = workloads.make_tree_inputs(8, 24, 3001, "f32", "star", a=-0.5, e=2.0, lam=0.2, seed=5,
                                   device=DEV)
    n, _ = _check(specv, x, 0)
    assert (n <= 1).all()


@pytest.mark.parametrize("S", [1, 2, 3, 4, 8, 13, 16])
def test_tree_every_cluster_size(specv, env_guard, S):
    os.environ["SPECV_CLUSTER_SIZE"] = str(S)
    x = workloads.make_tree_inputs(4, 7, 50000, "bf16", "kary:2", lam=0.25, seed=7, device=DEV)
    _check(specv, x, 0)
    x = workloads.make_tree_inputs(3, 5, 40001, "f32", "random:3", lam=0.5, seed=8, device=DEV)
    _check(specv, x, 1)  # rows off 16-byte boundaries


def test_tree_chain_matches_chain_verify(specv):
    """A chain-shaped tree is the chain verify step: same decisions as
    specv_verify on the same logits and uniforms (away from boundaries)."""
    w = workloads.WORKLOADS[3].scaled(B=16, V=8192)
    x = workloads.make_inputs(w, DEV)
    B, K = w.B, w.K
    parent = torch.arange(-1, K, dtype=torch.int32, device=DEV).repeat(B, 1).contiguous()
    drow = torch.arange(0, K + 1, dtype=torch.int32, device=DEV).repeat(B, 1)
    drow[:, K] = -1
    tokens = torch.zeros((B, K + 1), dtype=torch.int32, device=DEV)
    tokens[:, 1:] = x["draft_tokens"]
    ua = torch.zeros((B, K + 1), dtype=torch.float32, device=DEV)
    ua[:, 1:] = x["u_accept"]
    tt, tp, tn = specv.verify_tree(x["target_logits"], x["draft_logits"], parent,
                                   drow.contiguous(), tokens, ua, x["u_resample"], x["lam"])
    ct, cn = specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                          x["u_accept"], x["u_resample"], x["lam"])
    orc = oracle.verify(*[x[k].cpu() for k in ("target_logits", "draft_logits", "draft_tokens",
                                                "u_accept", "u_resample", "lam")])
    far = (orc.accept_margin >= BAND) & (orc.cdf_margin >= BAND)
    assert far.sum() >= B // 2
    np.testing.assert_array_equal(tn.cpu().numpy()[far], cn.cpu().numpy()[far])
    np.testing.assert_array_equal(tt.cpu().numpy()[far], ct.cpu().numpy()[far])


def test_tree_invalid_inputs(specv):
    x = workloads.make_tree_inputs(6, 6, 500, "f32", "kary:2", seed=9, device=DEV)
    x["parent"][1, 0] = 0          # root with a parent
    x["parent"][2, 5] = 5          # a node its own parent
    x["draft_row"][3, 1] = -1      # node 1 has children but no draft row
    x["tokens"][4, 3] = 500        # token outside the vocabulary
    x["lam"][5] = 2.0
    n, _ = _check(specv, x, 0)
    assert (n[1:] == -1).all() and n[0] >= 0
    with pytest.raises(ValueError):
        specv.verify_tree(*_args(x), mode=2)
