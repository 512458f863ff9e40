"""specv_verify_sharded_host on one GPU: a batch split into shards that run on
the same device (separate library streams and staging) gives, sequence for
sequence, the outputs of the whole batch in one call -- bit for bit when the
launch plan is pinned (cluster size and draw placement fixed, since the plan
otherwise depends on a shard's size) -- including a shard count above B
(empty shards).  Multi-device runs take the same path with other device
indices; every call of this suite has one GPU.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def specv():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    import speculative_decoding_verification_specv_gb300 as m
    m.load(build_if_missing=True)
    return m


@pytest.fixture
def pinned_plan():
    keys = ("SPECV_CLUSTER_SIZE", "SPECV_SAMPLE_SPLIT", "SPECV_ROWS_VARIANT")
    old = {k: os.environ.get(k) for k in keys}
    os.environ.update(SPECV_CLUSTER_SIZE="4", SPECV_SAMPLE_SPLIT="0", SPECV_ROWS_VARIANT="stream")
    yield
    for k, v in old.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def _host(x):
    out = {}
    for k, v in x.items():
        h = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
        h.copy_(v)
        out[k] = h
    return out


def _args(h):
    return (h["target_logits"], h["draft_logits"], h["draft_tokens"], h["u_accept"],
            h["u_resample"], h["lam"])


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["prob", "logit", "greedy"])
@pytest.mark.parametrize("shards", [2, 3, 8])
@pytest.mark.parametrize("B", [7, 2])
def test_sharded_equals_one_call(specv, pinned_plan, B, shards, mode):
    w = workloads.WORKLOADS[3].scaled(B=B)
    h = _host(workloads.make_inputs(w, "cuda:0", seed_offset=B))
    ref_t, ref_n = specv.verify_host(*_args(h), mode=mode, chunks=1)
    torch.cuda.synchronize()
    tok, n = specv.verify_sharded(*_args(h), devices=[0] * shards, mode=mode)
    assert torch.equal(tok, ref_t) and torch.equal(n, ref_n)
    # and the shards' outputs against the oracle
    if mode == 2:
        orc = oracle.verify_greedy(h["target_logits"], h["draft_logits"], h["draft_tokens"],
                                   h["lam"])
        _parity.compare_greedy(h, tok.numpy(), n.numpy(), orc)
    else:
        _parity.compare(h, mode, tok.numpy(), n.numpy(), _parity.run_oracle(h, mode))


def test_sharded_batched_workload_against_the_oracle(specv):
    """The batched 128K-vocabulary workload at B = 40 in 4 shards with the
    library's own plans (each shard its own plan): agreement with the oracle
    outside the decision band."""
    w = workloads.WORKLOADS[4].scaled(B=40)
    h = _host(workloads.make_inputs(w, "cuda:0"))
    tok, n = specv.verify_sharded(*_args(h), devices=[0, 0, 0, 0])
    rep = _parity.compare(h, 0, tok.numpy(), n.numpy(), _parity.run_oracle(h, 0))
    assert (n.numpy()[20:] == w.K).all()  # the drafted-equals-target half accepts everything
    print(rep)


def test_sharded_rejects_devices_that_do_not_exist(specv):
    w = workloads.WORKLOADS[1]
    h = _host(workloads.make_inputs(w, "cuda:0"))
    with pytest.raises(specv.SpecvError):
        specv.verify_sharded(*_args(h), devices=[0, torch.cuda.device_count()])
    with pytest.raises(specv.SpecvError):
        specv.verify_sharded(*_args(h), devices=[-1])
    assert torch.cuda.current_device() == 0
