"""GPU tests of the host-buffer entry point (specv_verify_host).

With one chunk the call runs the same launch plan as specv_verify on the
same batch, so its outputs must equal specv_verify's bit for bit.  With more
chunks each chunk is a smaller batch (possibly another plan and rounding
order of the row sums): decisions are compared with the oracle, exactly
outside the 1e-5 band of a decision or CDF boundary.  Greedy decisions do not
depend on the plan, so they must equal specv_verify's for any chunk count.
"""
import numpy as np
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


KEYS = ("target_logits", "draft_logits", "draft_tokens", "u_accept", "u_resample", "lam")


def _host(x, pinned=True):
    out = {}
    for k in KEYS:
        t = torch.empty(x[k].shape, dtype=x[k].dtype, pin_memory=pinned)
        t.copy_(x[k])
        out[k] = t
    return out


def _device_ref(specv, x, mode):
    tok, n = specv.verify(*(x[k] for k in KEYS), mode=mode)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), n.cpu().numpy()


def _host_run(specv, h, mode, chunks, stream=None):
    tok, n = specv.verify_host(*(h[k] for k in KEYS), mode=mode, chunks=chunks, stream=stream)
    torch.cuda.synchronize()
    return tok.numpy().copy(), n.numpy().copy()


SHAPES = [
    # (workload, overrides)
    (1, dict(B=5)),                        # V=1000 fp32
    (3, dict(B=12, V=32000)),              # bf16 rows
    (5, dict(B=3000)),                     # V=32: the tile kernels
    (1, dict(B=9, K=3, V=33)),             # rows off 16-byte boundaries
    (4, dict(B=7, K=2, V=50000)),
]


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"w{s[0]}-" + "-".join(
    f"{k}{v}" for k, v in s[1].items()))
def test_one_chunk_equals_device_verify(specv, shape, mode):
    cfg, kw = shape
    w = workloads.WORKLOADS[cfg].scaled(**kw)
    x = workloads.make_inputs(w, DEV)
    ref_tok, ref_n = _device_ref(specv, x, mode)
    tok, n = _host_run(specv, _host(x), mode, chunks=1)
    np.testing.assert_array_equal(n, ref_n)
    np.testing.assert_array_equal(tok, ref_tok)


@pytest.mark.parametrize("chunks", [0, 2, 5, 64])
@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"w{s[0]}-" + "-".join(
    f"{k}{v}" for k, v in s[1].items()))
def test_chunked_parity_with_oracle(specv, shape, mode, chunks):
    cfg, kw = shape
    w = workloads.WORKLOADS[cfg].scaled(**kw)
    if w.B * w.V > 2_000_000:
        w = w.scaled(B=max(1, 2_000_000 // w.V))  # keep the oracle to seconds
    x = workloads.make_inputs(w, DEV, seed_offset=chunks)
    tok, n = _host_run(specv, _host(x), mode, chunks)
    xh = _parity.to_host(x)
    rep = _parity.compare(xh, mode, tok, n, _parity.run_oracle(xh, mode))
    assert rep["exact"] + rep["near_band"] == rep["sequences"]


@pytest.mark.parametrize("chunks", [0, 1, 3, 64])
def test_greedy_any_chunks_equals_device_verify(specv, chunks):
    for cfg, kw in SHAPES:
        w = workloads.WORKLOADS[cfg].scaled(**kw)
        x = workloads.make_inputs(w, DEV)
        ref_tok, ref_n = _device_ref(specv, x, 2)
        tok, n = _host_run(specv, _host(x), 2, chunks)
        np.testing.assert_array_equal(n, ref_n)
        np.testing.assert_array_equal(tok, ref_tok)


def test_back_to_back_calls_and_staging_growth(specv):
    """Three calls queued without a synchronisation in between, the second on
    a larger batch (the staging grows while the first call may still run):
    each call's outputs are its own inputs' results."""
    ws = [workloads.WORKLOADS[1].scaled(B=6, V=4096), workloads.WORKLOADS[4].scaled(B=40, V=8192),
          workloads.WORKLOADS[1].scaled(B=6, V=4096)]
    xs = [workloads.make_inputs(w, DEV, seed_offset=i) for i, w in enumerate(ws)]
    refs = [_device_ref(specv, x, 0) for x in xs]
    hs = [_host(x) for x in xs]
    outs = [specv.verify_host(*(h[k] for k in KEYS), chunks=c) for h, c in zip(hs, (3, 0, 2))]
    torch.cuda.synchronize()
    for i, ((tok, n), (ref_tok, ref_n)) in enumerate(zip(outs, refs)):
        same = (n.numpy() == ref_n) & (tok.numpy() == ref_tok).all(axis=1)
        if not same.all():  # another plan per chunk: differences only at boundaries
            xh = _parity.to_host(xs[i])
            _parity.compare(xh, 0, tok.numpy(), n.numpy(), _parity.run_oracle(xh, 0))


def test_pageable_inputs_and_side_stream(specv):
    w = workloads.WORKLOADS[3].scaled(B=5, V=20000)
    x = workloads.make_inputs(w, DEV)
    ref_tok, ref_n = _device_ref(specv, x, 1)
    s = torch.cuda.Stream()
    tok, n = _host_run(specv, _host(x, pinned=False), 1, chunks=1, stream=s)
    np.testing.assert_array_equal(n, ref_n)
    np.testing.assert_array_equal(tok, ref_tok)


def test_invalid_inputs_reported_per_sequence(specv):
    w = workloads.WORKLOADS[1].scaled(B=8, V=700)
    x = workloads.make_inputs(w, DEV)
    x["draft_tokens"][2, 1] = 700
    x["lam"][5] = float("nan")
    h = _host(x)
    for chunks in (1, 3, 8):
        tok, n = _host_run(specv, h, 0, chunks)
        assert n[2] == -1 and n[5] == -1 and (tok[[2, 5]] == -1).all()
        assert (np.delete(n, [2, 5]) >= 0).all()


def test_refused_under_graph_capture(specv):
    w = workloads.WORKLOADS[1].scaled(B=2, V=512)
    h = _host(workloads.make_inputs(w, DEV))
    out_tok = torch.empty((2, w.K + 1), dtype=torch.int32, pin_memory=True)
    out_n = torch.empty((2,), dtype=torch.int32, pin_memory=True)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(specv.SpecvError) as ei:
        with torch.cuda.graph(g, stream=s):
            specv.verify_host(*(h[k] for k in KEYS), out_tokens=out_tok, out_n_accepted=out_n)
    assert ei.value.status == 2


def test_full_size_batched_fp32(specv):
    """B=256, K=8, V=128256 fp32 (2.2 GB of pinned logits) with the automatic
    chunking: equal to specv_verify except in boundary cases, which the oracle
    must confirm; 16 sampled sequences against the oracle as well."""
    w = workloads.WORKLOADS[4]
    x = workloads.make_inputs(w, DEV)
    ref_tok, ref_n = _device_ref(specv, x, 0)
    h = _host(x)
    del x["target_logits"], x["draft_logits"]
    tok, n = _host_run(specv, h, 0, chunks=0)
    differ = np.nonzero((n != ref_n) | (tok != ref_tok).any(axis=1))[0].tolist()
    seqs = sorted(set(differ) | set(range(0, 256, 16)))
    orc = _parity.run_oracle(h, 0, seqs)
    _parity.compare(h, 0, tok, n, orc, seqs)
    assert len(differ) <= 4, differ


def _early_exit_run(specv, h, mode):
    tok, n, h2d, d2h = specv.verify_host_early_exit(*(h[k] for k in KEYS), mode=mode)
    torch.cuda.synchronize()
    K = h["draft_tokens"].shape[1]
    B = h["draft_tokens"].shape[0]
    assert B * (K + 2) * 4 <= d2h <= B * (K + 2) * 4 + K * B  # outputs, then one flag byte a level
    return tok.numpy().copy(), n.numpy().copy(), h2d


EE_SHAPES = SHAPES + [(4, dict(B=24, K=8, V=128256)),   # half the batch drafts the target
                      (3, dict(B=6))]                    # Qwen-shaped bf16 rows


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["prob", "logit", "greedy"])
@pytest.mark.parametrize("shape", EE_SHAPES, ids=lambda s: f"w{s[0]}-" + "-".join(
    f"{k}{v}" for k, v in s[1].items()))
def test_early_exit_host_call_equals_device_verify(specv, shape, mode):
    """specv_verify_host_early_exit copies position by position and stops at a
    sequence's first clear rejection: its outputs equal specv_verify's bit for
    bit (the rows it leaves out are never read for an output), it copies no
    more than every row and at least every row the outputs depend on.  The
    staging first holds another batch's rows (a call on other inputs), so the
    rows left out are stale, not zero."""
    cfg, kw = shape
    w = workloads.WORKLOADS[cfg].scaled(**kw)
    other = workloads.make_inputs(w, DEV, seed_offset=5)
    _host_run(specv, _host(other), mode, chunks=1)  # stale rows in the staging
    x = workloads.make_inputs(w, DEV)
    ref_tok, ref_n = _device_ref(specv, x, mode)
    tok, n, h2d = _early_exit_run(specv, _host(x), mode)
    np.testing.assert_array_equal(n, ref_n)
    np.testing.assert_array_equal(tok, ref_tok)
    s = w.elem_bytes
    every = (2 * w.K + 1) * w.B * w.V * s + 2 * w.B * w.K * 4 + 2 * w.B * 4
    rows_needed = sum(2 * min(int(k) + 1, w.K) + (int(k) == w.K) for k in n)
    assert rows_needed * w.V * s <= h2d <= every
    print(f"{shape} mode={mode}: copied {h2d / every:.3f} of every row")


def test_release_stream_frees_and_reallocates(specv):
    """specv_release_stream frees a stream's scratch (grown twice, so with
    superseded buffers) and staging; later calls on the stream allocate afresh
    and give the same outputs.  Under capture it refuses."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    outs = []
    for B in (4, 9, 17):  # the scratch grows
        w = workloads.WORKLOADS[3].scaled(B=B)
        x = workloads.make_inputs(w, DEV)
        with torch.cuda.stream(s):
            outs.append([t.clone() for t in specv.verify(*(x[k] for k in KEYS), stream=s)])
    h = _host(x)
    with torch.cuda.stream(s):
        ref_h = specv.verify_host(*(h[k] for k in KEYS), chunks=1, stream=s)
        s.synchronize()  # the host outputs are complete only once the stream is
        ref_h = [t.clone() for t in ref_h]
        specv.verify_host_early_exit(*(h[k] for k in KEYS), stream=s)
    s.synchronize()
    before = torch.cuda.mem_get_info()[0]
    with torch.cuda.stream(s):
        specv.release_stream(s)
    after = torch.cuda.mem_get_info()[0]
    assert after >= before  # the staging and scratch went back to the device
    with torch.cuda.stream(s):
        again = specv.verify(*(x[k] for k in KEYS), stream=s)
        again_h = specv.verify_host(*(h[k] for k in KEYS), chunks=1, stream=s)
    s.synchronize()
    assert torch.equal(again[0], outs[-1][0]) and torch.equal(again[1], outs[-1][1])
    assert torch.equal(again_h[0], ref_h[0]) and torch.equal(again_h[1], ref_h[1])
    g = torch.cuda.CUDAGraph()
    s2 = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s2):
        st = specv.raw_call("specv_release_stream", s2.cuda_stream)
    assert st == 2


DIRECT_SHAPES = [
    (4, dict(B=24, K=8, V=128256), True),   # streaming kernel in both calls: bit-equal
    (3, dict(B=8), True),
    (1, dict(B=9, K=3, V=33), True),        # rows off 16-byte boundaries: generic tile kernel
    (5, dict(B=3000), False),               # short rows: no TMA tile kernel on host memory
    (2, dict(), False),                     # B = 1: no resident (TMA-staged) kernel either
]


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["prob", "logit", "greedy"])
@pytest.mark.parametrize("shape", DIRECT_SHAPES, ids=lambda s: f"w{s[0]}-" + "-".join(
    f"{k}{v}" for k, v in s[1].items()))
def test_direct_host_call(specv, shape, mode):
    """specv_verify_host_direct: the kernels read the page-locked host inputs
    and write the host outputs in place.  Where the device call plans the same
    kernel the outputs are equal bit for bit; elsewhere (the kernels that stage
    rows by bulk copy are not planned on host memory) they agree with the
    oracle outside the decision band."""
    cfg, kw, same_plan = shape
    w = workloads.WORKLOADS[cfg].scaled(**kw)
    x = workloads.make_inputs(w, DEV)
    h = _host(x)
    tok, n = specv.verify_host_direct(*(h[k] for k in KEYS), mode=mode)
    torch.cuda.synchronize()
    tok, n = tok.numpy().copy(), n.numpy().copy()
    if same_plan:
        ref_tok, ref_n = _device_ref(specv, x, mode)
        np.testing.assert_array_equal(n, ref_n)
        np.testing.assert_array_equal(tok, ref_tok)
    xh = _parity.to_host(x)
    if mode == 2:
        import oracle
        orc = oracle.verify_greedy(xh["target_logits"], xh["draft_logits"], xh["draft_tokens"],
                                   xh["lam"])
        _parity.compare_greedy(xh, tok, n, orc)
    else:
        _parity.compare(xh, mode, tok, n, _parity.run_oracle(xh, mode))


def test_direct_host_call_pageable_or_refused(specv):
    """Pageable host tensors: read in place where the device reads pageable
    memory, refused with SPECV_ERR_UNSUPPORTED (nothing launched) elsewhere."""
    w = workloads.WORKLOADS[3].scaled(B=4)
    x = workloads.make_inputs(w, DEV)
    h = _host(x, pinned=False)
    ref_tok, ref_n = _device_ref(specv, x, 0)
    out_t = torch.empty((w.B, w.K + 1), dtype=torch.int32)
    out_n = torch.empty((w.B,), dtype=torch.int32)
    try:
        specv.verify_host_direct(*(h[k] for k in KEYS), out_tokens=out_t, out_n_accepted=out_n)
    except specv.SpecvError as e:
        assert e.status == 2
        return
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out_n.numpy(), ref_n)
    np.testing.assert_array_equal(out_t.numpy(), ref_tok)
