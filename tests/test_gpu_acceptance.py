"""GPU parity of specv_acceptance_rates: alpha[b][i] = sum_v min(p~_v, q_v) of
every drafted position against the oracle's fp64 value, within the
probability tolerance of the parity contract (1e-5 for fp32 logits, 2e-3 for
bf16), plus its invariants (alpha = 1 when the draft equals the target or, in
probability mode, when lambda = 1), NaN for invalid lambda, and the host
controller fed from the device statistics."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

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
    old = os.environ.get("SPECV_CLUSTER_SIZE")
    yield
    if old is None:
        os.environ.pop("SPECV_CLUSTER_SIZE", None)
    else:
        os.environ["SPECV_CLUSTER_SIZE"] = old


def _check(specv, x, mode, seqs=None):
    alpha = specv.acceptance_rates(x["target_logits"], x["draft_logits"], x["lam"], mode=mode)
    torch.cuda.synchronize()
    got = alpha.cpu().numpy().astype(np.float64)
    sub = x if seqs is None else {k: v.index_select(0, torch.as_tensor(seqs, device=v.device))
                                  for k, v in x.items()}
    r = oracle.verify(sub["target_logits"], sub["draft_logits"], sub["draft_tokens"],
                      sub["u_accept"], sub["u_resample"], sub["lam"], mode=mode)
    ref = r.alpha
    if seqs is not None:
        got = got[seqs]
    tol = 2e-3 if x["target_logits"].dtype == torch.bfloat16 else 1e-5
    ok = ~np.isnan(ref)
    err = np.abs(got[ok] - ref[ok])
    assert err.max(initial=0.0) <= tol, (err.max(), tol)
    assert np.isnan(got[~ok]).all()
    return got, float(err.max(initial=0.0))


SMALL = {
    1: workloads.WORKLOADS[1],
    2: workloads.WORKLOADS[2],
    3: workloads.WORKLOADS[3].scaled(B=8),
    4: workloads.WORKLOADS[4].scaled(B=8),
    5: workloads.WORKLOADS[5].scaled(B=2000),
}


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_acceptance_rates_workloads(specv, cfg, mode):
    w = SMALL[cfg]
    x = workloads.make_inputs(w, DEV)
    got, err = _check(specv, x, mode)
    print(f"alpha workload {cfg} mode={mode}: max |err| {err:.2e}, mean alpha {np.nanmean(got):.4f}")


def test_acceptance_rates_full_size_sampled(specv):
    w = workloads.WORKLOADS[4]
    x = workloads.make_inputs(w, DEV)
    got, _ = _check(specv, x, 0, seqs=[0, 1, 77, 128, 200, 255])
    full = specv.acceptance_rates(x["target_logits"], x["draft_logits"], x["lam"]).cpu().numpy()
    # the second half drafts with the target itself: alpha = 1 up to round-off
    assert np.abs(full[128:] - 1.0).max() < 1e-5


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
def test_acceptance_rates_every_cluster_size(specv, env_guard, S):
    os.environ["SPECV_CLUSTER_SIZE"] = str(S)
    w = workloads.WORKLOADS[3].scaled(B=3, V=40000)
    x = workloads.make_inputs(w, DEV)
    _check(specv, x, 1)
    w = workloads.WORKLOADS[4].scaled(B=2, K=3, V=65537)  # rows off 16-byte boundaries
    x = workloads.make_inputs(w, DEV)
    _check(specv, x, 0)


@pytest.mark.parametrize("shape", [(3, 1, 1001, "f32"), (2, 33, 515, "bf16"), (5, 3, 33, "f32"),
                                   (1, 1, 1, "f32"), (4, 2, 131071, "f32")],
                         ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}")
def test_acceptance_rates_ragged_shapes(specv, shape):
    B, K, V, dt = shape
    w = workloads.Workload("ragged", B, K, V, dt, "corr:2.0:0.8:1.0", (0.35,), 9)
    x = workloads.make_inputs(w, DEV)
    for mode in (0, 1):
        _check(specv, x, mode)


def test_acceptance_rates_invariants_and_errors(specv):
    w = workloads.WORKLOADS[3].scaled(B=5, V=3001)
    x = workloads.make_inputs(w, DEV)
    same = dict(x)
    same["draft_logits"] = x["target_logits"][:, :w.K].contiguous()
    for mode in (0, 1):
        a = specv.acceptance_rates(same["target_logits"], same["draft_logits"], same["lam"],
                                   mode=mode)
        assert (a.cpu() - 1.0).abs().max() < 1e-5
    one = torch.ones_like(x["lam"])
    a = specv.acceptance_rates(x["target_logits"], x["draft_logits"], one, mode=0)
    assert (a.cpu() - 1.0).abs().max() < 1e-5  # p~ = q
    bad = x["lam"].clone()
    bad[1] = 1.5
    bad[3] = float("nan")
    a = specv.acceptance_rates(x["target_logits"], x["draft_logits"], bad, mode=0).cpu()
    assert torch.isnan(a[1]).all() and torch.isnan(a[3]).all() and not torch.isnan(a[0]).any()
    with pytest.raises(ValueError):
        specv.acceptance_rates(x["target_logits"], x["draft_logits"], x["lam"], mode=2)
    st = specv.raw_call("specv_acceptance_rates", x["target_logits"].data_ptr(),
                        x["draft_logits"].data_ptr(), x["lam"].data_ptr(), w.B, w.K, w.V, 1, 2,
                        x["u_accept"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 2  # greedy: unsupported


def test_adaptive_k_from_device_statistics(specv):
    """The controller on the device's acceptance probabilities: the noisy draft
    (low alpha) gets a shorter draft than the faithful one (alpha near 1)."""
    w = workloads.WORKLOADS[4].scaled(B=16, V=32000)
    x = workloads.make_inputs(w, DEV)
    a = specv.acceptance_rates(x["target_logits"], x["draft_logits"], x["lam"])
    lo = specv.AdaptiveK(cost_draft=0.2, cost_verify_fixed=3.0, cost_verify_per_token=0.02)
    hi = specv.AdaptiveK(cost_draft=0.2, cost_verify_fixed=3.0, cost_verify_per_token=0.02)
    for _ in range(10):
        k_lo = lo.update(a[:8])     # corr half
        k_hi = hi.update(a[8:])     # draft == target half
    assert hi.alpha > 0.999 and lo.alpha < hi.alpha
    assert k_hi == 16 and k_lo <= k_hi
