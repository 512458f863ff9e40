"""GPU parity: the CUDA verify step (through the C ABI) against the fp64 oracle.

Decisions (n_accepted and every emitted token) must be bit-exact except where
a uniform lies within 1e-5 of a decision or CDF boundary; those sequences are
counted and must still hold a valid outcome.  The probabilities p~(x_i) and
q(x_i) the kernels computed must match the oracle within 1e-5 (fp32 logits)
or 2e-3 (bf16 logits).
"""
import os

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


@pytest.fixture
def cluster_env():
    keys = ("SPECV_CLUSTER_SIZE", "SPECV_ROWS_VARIANT", "SPECV_SAMPLE_SPLIT", "SPECV_EARLY_EXIT")
    old = {k: os.environ.get(k) for k in keys}
    yield
    for k, v in old.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def _set_variant(variant):
    """Force a row kernel: "stream" (the streaming kernel) or "resident"."""
    os.environ["SPECV_ROWS_VARIANT"] = variant


def _run(specv, x, mode, debug=True):
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    tok, n = specv.verify(*args, mode=mode)
    dbg = specv.verify_debug(*args, mode=mode) if debug else None
    torch.cuda.synchronize()
    if dbg is not None:
        # the debug entry point runs the same kernels: same decisions
        assert torch.equal(dbg["tokens"], tok) and torch.equal(dbg["n_accepted"], n)
    return tok.cpu().numpy(), n.cpu().numpy(), dbg


def _check(specv, x, mode, seqs=None, debug=True):
    tok, n, dbg = _run(specv, x, mode, debug)
    xh = _parity.to_host(x)
    orc = _parity.run_oracle(xh, mode, seqs)
    rep = _parity.compare(xh, mode, tok, n, orc, seqs)
    if dbg is not None:
        rep.update(_parity.check_probabilities(xh, mode, dbg, orc, seqs))
    return rep, tok, n


SMALL = {
    1: workloads.WORKLOADS[1],
    2: workloads.WORKLOADS[2],
    3: workloads.WORKLOADS[3],
    4: workloads.WORKLOADS[4].scaled(B=16),
    5: workloads.WORKLOADS[5].scaled(B=50_000),
}


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_parity_workloads(specv, cfg, mode):
    w = SMALL[cfg]
    x = workloads.make_inputs(w, DEV)
    rep, tok, n = _check(specv, x, mode)
    print(f"workload {cfg} ({w.name}, B={w.B}) mode={mode}: {rep}")
    assert rep["exact"] + rep["near_band"] == rep["sequences"]


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_whole_row_probabilities(specv, cfg, mode):
    """Every entry of p~ and q (not only at the drafted tokens), as implied by
    the kernels' row log-normalisers, against the oracle's fp64 rows within
    1e-5 (fp32 logits) / 2e-3 (bf16 logits); two sequences per workload."""
    w = SMALL[cfg]
    x = workloads.make_inputs(w, DEV)
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    dbg = specv.verify_debug(*args, mode=mode)
    torch.cuda.synchronize()
    xh = _parity.to_host(x)
    rep = _parity.check_rows(xh, mode, dbg, seqs=[0, w.B - 1])
    print(f"workload {cfg} mode={mode}: {rep}")


@pytest.mark.parametrize("early", ["0", "1"], ids=["all-rows", "early-exit"])
@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
def test_parity_full_size_batched_fp32_sampled(specv, cluster_env, mode, early):
    """B=256, K=8, V=128256 fp32 as benchmarked; the oracle checks 32 sampled
    sequences, and every drafted-equals-target sequence must accept all K.
    With SPECV_EARLY_EXIT=1 positions after a published rejection skip their
    rows: the outputs must not change."""
    os.environ["SPECV_EARLY_EXIT"] = early
    w = workloads.WORKLOADS[4]
    x = workloads.make_inputs(w, DEV)
    seqs = list(range(0, 128, 8)) + list(range(128, 256, 8))
    rep, tok, n = _check(specv, x, mode, seqs=seqs)
    print(f"full-size batched fp32 mode={mode}: {rep}")
    assert (n[128:] == w.K).all()
    assert ((tok[128:, :w.K] == x["draft_tokens"][128:].cpu().numpy())).all()
    assert ((tok[128:, w.K] >= 0) & (tok[128:, w.K] < w.V)).all()


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
def test_parity_full_size_exactness_workload(specv, mode):
    w = workloads.WORKLOADS[5]
    x = workloads.make_inputs(w, DEV)
    rep, _, _ = _check(specv, x, mode, debug=False)
    print(f"full-size exactness workload mode={mode}: {rep}")


@pytest.mark.parametrize("S", [1, 2, 3, 4, 6, 8, 15, 16])
@pytest.mark.parametrize("variant", ["stream", "resident"])
def test_every_cluster_size(specv, cluster_env, variant, S):
    os.environ["SPECV_CLUSTER_SIZE"] = str(S)
    _set_variant(variant)
    cases = ((workloads.WORKLOADS[3].scaled(B=4), 0),
             (workloads.WORKLOADS[1].scaled(B=3, K=3, V=50000), 1),
             (workloads.WORKLOADS[4].scaled(B=2, K=2, V=4096), 0))
    ran = 0
    for w, mode in cases:
        dt = 1 if w.dtype == "bf16" else 0
        try:
            plan = specv.plan(w.B, w.K, w.V, dt)
        except specv.SpecvError:
            continue  # this slice does not fit shared memory at this cluster size
        assert plan["cluster"] == S and plan["kernel"] == "rows-" + variant
        x = workloads.make_inputs(w, DEV)
        rep, _, _ = _check(specv, x, mode)
        ran += 1
        print(f"{variant} S={S} {w.name} V={w.V}: {rep}")
    assert ran >= 1


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_streaming_kernel_on_workloads(specv, cluster_env, cfg, mode):
    _set_variant("stream")
    w = SMALL[cfg]
    x = workloads.make_inputs(w, DEV)
    assert specv.plan(w.B, w.K, w.V, 1 if w.dtype == "bf16" else 0)["kernel"] == "rows-stream"
    rep, _, _ = _check(specv, x, mode)
    print(f"streaming kernel, workload {cfg}: {rep}")


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("V,dt", [(300000, "f32"), (300001, "f32"), (600000, "bf16")])
def test_long_slices_multi_tile_segments(specv, cluster_env, V, dt, mode):
    """One CTA per row and slices of 75000 groups: more groups than the sampler's
    segment table holds in single tiles, so every segment spans two tiles.  Half
    the sequences accept every draft (bonus rows sampled from the segment
    statistics of the first pass), the rest reject (residual walk)."""
    os.environ["SPECV_CLUSTER_SIZE"] = "1"
    _set_variant("stream")
    w = workloads.Workload("long-slices", 6, 3, V, dt, "half_equal:3.0:0.85:1.0", (0.2,), 11)
    plan = specv.plan(w.B, w.K, w.V, 1 if dt == "bf16" else 0, mode)
    assert plan["kernel"] == "rows-stream" and plan["cluster"] == 1
    x = workloads.make_inputs(w, DEV)
    rep, _, n = _check(specv, x, mode)
    assert (n == w.K).any() and (n < w.K).any()
    print(f"V={V} {dt} mode={mode}: {rep}")


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("split", ["0", "1"], ids=["fused", "split"])
@pytest.mark.parametrize("shape", [(8, 5, 152064, "bf16", "rho:3.0:0.5:0.95"),
                                   (16, 8, 128256, "f32", "half_equal:3.0:0.85:1.0"),
                                   (5, 3, 1001, "f32", "corr:2.0:0.8:1.0"),
                                   (3, 33, 515, "bf16", "corr:3.0:0.9:0.7"),
                                   (6, 4, 300001, "f32", "half_equal:3.0:0.85:1.0")],
                         ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}")
def test_token_draws_in_one_or_two_launches(specv, cluster_env, shape, split, mode):
    """The streaming kernel's token draws in the statistics launch (fused) or in
    a second launch with a wider cluster per sequence (split): both give the
    oracle's decisions, bonus rows included."""
    _set_variant("stream")
    os.environ["SPECV_SAMPLE_SPLIT"] = split
    B, K, V, dt, st = shape
    w = workloads.Workload("split", B, K, V, dt, st, (0.3,), 17)
    x = workloads.make_inputs(w, DEV)
    rep, _, n = _check(specv, x, mode)
    print(f"{shape} split={split} mode={mode}: {rep}")


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("V,dt", [(64, "f32"), (1000, "bf16")])
def test_maximum_draft_length(specv, V, dt, mode):
    """K = 4096, the largest draft the boundary accepts: 4097 positions per
    sequence.  The second sequence drafts the target itself, so all 4096 drafts
    pass and the bonus row is drawn; the first rejects early."""
    w = workloads.Workload("kmax", 2, 4096, V, dt, "half_equal:2.0:0.9:0.5", (0.3,), 31)
    x = workloads.make_inputs(w, DEV)
    rep, tok, n = _check(specv, x, mode, debug=False)
    print(f"K=4096 V={V} {dt} mode={mode}: {rep}, n={n.tolist()}")
    assert n[1] == 4096 and (tok[1, :4096] == x["draft_tokens"][1].cpu().numpy()).all()
    assert 0 <= tok[1, 4096] < V


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("shape", [(400, 3, 4099, "f32", "corr:3.0:0.85:1.0"),
                                   (96, 8, 65536, "bf16", "half_equal:3.0:0.85:1.0"),
                                   (200, 6, 20000, "f32", "rho:3.0:0.5:0.95")],
                         ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}")
def test_early_exit_parity(specv, cluster_env, shape, mode):
    """Early exit (SPECV_EARLY_EXIT=1): grids of several waves, position-major,
    positions after a published rejection read nothing.  Every sequence agrees
    with the oracle, and with the all-rows run bit for bit."""
    B, K, V, dt, st = shape
    w = workloads.Workload("early", B, K, V, dt, st, (0.3,), 37)
    x = workloads.make_inputs(w, DEV)
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    os.environ["SPECV_EARLY_EXIT"] = "0"
    t0, n0 = specv.verify(*args, mode=mode)
    os.environ["SPECV_EARLY_EXIT"] = "1"
    assert specv.plan(B, K, V, 1 if dt == "bf16" else 0, mode)["kernel"] == "rows-stream"
    t1, n1 = specv.verify(*args, mode=mode)
    t2, n2 = specv.verify(*args, mode=mode)  # the scratch words were left at zero
    torch.cuda.synchronize()
    assert torch.equal(t0, t1) and torch.equal(n0, n1)
    assert torch.equal(t1, t2) and torch.equal(n1, n2)
    rep, _, _ = _check(specv, x, mode, debug=False)
    print(f"{shape} mode={mode}: {rep}")


RAGGED = [
    # (B, K, V, dtype, structure)
    (3, 1, 1001, "f32", "corr:2.0:0.8:1.0"),       # rows kernel, unaligned rows
    (2, 33, 515, "bf16", "corr:3.0:0.9:0.7"),      # K crosses one warp of positions
    (5, 3, 33, "f32", "corr:2.0:0.8:1.0"),         # tile kernel, V just over a warp
    (41, 4, 32, "f32", "broadcast:1.5"),           # tile kernel, ragged last tile
    (7, 2, 257, "bf16", "corr:3.0:0.9:0.7"),       # first V past the tile kernel
    (9, 2, 256, "bf16", "corr:3.0:0.9:0.7"),       # last V of the tile kernel
    (2, 64, 4099, "bf16", "rho:3.0:0.5:0.95"),     # many positions, odd V
    (1, 1, 1, "f32", "corr:2.0:0.8:1.0"),          # V = 1: certain tokens
    (3, 2, 2, "f32", "corr:2.0:0.8:1.0"),
    (1, 300, 3, "f32", "corr:2.0:0.8:1.0"),        # long draft, tiny vocabulary
    (2, 4, 131071, "f32", "corr:3.0:0.85:1.0"),    # odd large V, fp32
]


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}")
def test_ragged_shapes(specv, shape, mode):
    B, K, V, dt, st = shape
    w = workloads.Workload("ragged", B, K, V, dt, st, (0.35,), 9)
    x = workloads.make_inputs(w, DEV)
    rep, _, _ = _check(specv, x, mode)
    print(f"{shape} mode={mode} plan={specv.plan(B, K, V, 1 if dt == 'bf16' else 0, mode)}: {rep}")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("V", [24, 1000, 20000])
def test_misaligned_base_pointers(specv, dt, V):
    """Inputs that start one element past a 16-byte boundary."""
    w = workloads.Workload("misaligned", 3, 3, V, dt, "corr:2.0:0.8:1.0", (0.3,), 8)
    x = workloads.make_inputs(w, DEV)
    for key in ("target_logits", "draft_logits"):
        t = x[key]
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
        v = buf[1:].view(t.shape)
        v.copy_(t)
        assert v.data_ptr() % 16 != 0 and v.is_contiguous()
        x[key] = v
    _check(specv, x, 0)


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("V", [32, 3001, 128256])
def test_identical_draft_accepts_all(specv, mode, V):
    w = workloads.WORKLOADS[4].scaled(B=6, V=V)
    x = workloads.make_inputs(w, DEV)
    x["draft_logits"] = x["target_logits"][:, :w.K].contiguous()
    for lam in (0.0, 0.2, 1.0):
        x["lam"] = torch.full((w.B,), lam, dtype=torch.float32, device=DEV)
        tok, n, _ = _run(specv, x, mode, debug=False)
        assert (n == w.K).all(), (lam, n)
        assert (tok[:, :w.K] == x["draft_tokens"].cpu().numpy()).all()


def test_lambda_one_and_zero_uniforms_accept(specv):
    w = workloads.WORKLOADS[3].scaled(B=4, V=5003)
    x = workloads.make_inputs(w, DEV, lam=1.0)
    _, n, _ = _run(specv, x, 0, debug=False)
    assert (n == w.K).all()
    x = workloads.make_inputs(w, DEV)
    x["u_accept"].zero_()
    for mode in (0, 1):
        _, n, _ = _run(specv, x, mode, debug=False)
        assert (n == w.K).all()


@pytest.mark.parametrize("V", [32, 4099])
def test_invalid_inputs_give_minus_one(specv, V):
    w = workloads.WORKLOADS[1].scaled(B=5, V=V)
    x = workloads.make_inputs(w, DEV)
    x["draft_tokens"][1, 2] = V          # out of range
    x["draft_tokens"][2, 0] = -3         # negative
    x["lam"][3] = 1.5                    # not a convex weight
    x["lam"][4] = float("nan")
    tok, n, _ = _run(specv, x, 0, debug=False)
    for b in (1, 2, 3, 4):
        assert n[b] == -1 and (tok[b] == -1).all()
    assert n[0] >= 0
    xh = _parity.to_host(x)
    orc = _parity.run_oracle(xh, 0)
    _parity.compare(xh, 0, tok, n, orc)


def test_deterministic_and_stream_ordered(specv):
    w = workloads.WORKLOADS[3].scaled(B=8)
    x = workloads.make_inputs(w, DEV)
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    t0, n0 = specv.verify(*args)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        t1, n1 = specv.verify(*args, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(t0, t1) and torch.equal(n0, n1)


def test_binding_rejects_bad_tensors(specv):
    w = workloads.WORKLOADS[1]
    x = workloads.make_inputs(w, DEV)
    with pytest.raises(TypeError):
        specv.verify(x["target_logits"].double(), x["draft_logits"].double(), x["draft_tokens"],
                     x["u_accept"], x["u_resample"], x["lam"])
    with pytest.raises(ValueError):
        specv.verify(x["target_logits"], x["draft_logits"][:, :2].contiguous(),
                     x["draft_tokens"], x["u_accept"], x["u_resample"], x["lam"])
    with pytest.raises(ValueError):
        cpu = {k: v.cpu() for k, v in x.items()}
        specv.verify(cpu["target_logits"], cpu["draft_logits"], cpu["draft_tokens"],
                     cpu["u_accept"], cpu["u_resample"], cpu["lam"])


def test_streams_and_graph_capture_share_nothing_wrongly(specv):
    """Per-stream scratch: concurrent calls on two streams, a graph captured on
    a stream that already has scratch, and one captured on a fresh stream
    (stream-ordered scratch inside the graph) all give the eager results."""
    w = workloads.WORKLOADS[3].scaled(B=6)
    xs = [workloads.make_inputs(w, DEV, seed_offset=k) for k in range(2)]
    ref = []
    for x in xs:
        t, n = specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                            x["u_accept"], x["u_resample"], x["lam"])
        ref.append((t.clone(), n.clone()))
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for k, s in enumerate((s1, s2)):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            x = xs[k]
            outs.append(specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                                     x["u_accept"], x["u_resample"], x["lam"], stream=s))
    torch.cuda.synchronize()
    for (t, n), (rt, rn) in zip(outs, ref):
        assert torch.equal(t, rt) and torch.equal(n, rn)
    for warm in (True, False):
        x = xs[0]
        tok = torch.empty_like(ref[0][0])
        nn = torch.empty_like(ref[0][1])
        s = torch.cuda.Stream()
        if warm:  # the stream gets its scratch before the capture
            with torch.cuda.stream(s):
                specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                             x["u_accept"], x["u_resample"], x["lam"], out_tokens=tok,
                             out_n_accepted=nn, stream=s)
            s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
                         x["u_resample"], x["lam"], out_tokens=tok, out_n_accepted=nn,
                         stream=torch.cuda.current_stream())
        for _ in range(3):
            tok.fill_(-9)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(tok, ref[0][0]) and torch.equal(nn, ref[0][1])


SEQ_SHAPES = [
    # (B, K, V, dtype, structure): grids of about one wave with one cluster per sequence
    (32, 5, 152064, "bf16", "rho:3.0:0.5:0.95"),        # the Qwen-shaped workload
    (38, 3, 65536, "bf16", "half_equal:3.0:0.85:1.0"),  # half the sequences draw the bonus
    (20, 12, 65536, "f32", "corr:3.0:0.85:1.0"),
    (19, 32, 32768, "bf16", "half_equal:3.0:0.9:0.5"),  # 33 positions: more than a warp's lanes
    (24, 6, 40001, "bf16", "corr:2.0:0.8:1.0"),         # rows off 16-byte boundaries
    (30, 4, 40001, "f32", "half_equal:3.0:0.85:1.0"),
    (32, 2, 4099 * 8, "f32", "corr:2.0:0.8:1.0"),       # parts ending inside the bonus row
]


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("shape", SEQ_SHAPES, ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}")
def test_sequence_cluster_kernel(specv, cluster_env, shape, mode):
    """One cluster per sequence: every position streamed, decided and the token
    drawn in one launch; decisions and probabilities against the oracle."""
    B, K, V, dt, st = shape
    plan = specv.plan(B, K, V, 1 if dt == "bf16" else 0, mode)
    assert plan["kernel"] == "rows-seq" and plan["workspace_bytes"] == 0, plan
    w = workloads.Workload("seq", B, K, V, dt, st, ("uniform", 0.0, 0.6), 43)
    x = workloads.make_inputs(w, DEV)
    rep, tok, n = _check(specv, x, mode)
    if st.startswith("half_equal"):
        assert (n[B // 2:] == K).all()
    print(f"{shape} mode={mode} plan={plan}: {rep}")


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
def test_sequence_cluster_kernel_whole_rows_and_invalid_inputs(specv, mode):
    w = workloads.Workload("seq", 38, 3, 65536, "bf16", "corr:3.0:0.85:1.0", (0.3,), 44)
    x = workloads.make_inputs(w, DEV)
    x["draft_tokens"][1, 2] = w.V
    x["lam"][3] = float("nan")
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    dbg = specv.verify_debug(*args, mode=mode)
    torch.cuda.synchronize()
    n = dbg["n_accepted"].cpu().numpy()
    tok = dbg["tokens"].cpu().numpy()
    assert n[1] == -1 and n[3] == -1 and (tok[[1, 3]] == -1).all()
    xh = _parity.to_host(x)
    _parity.compare(xh, mode, tok, n, _parity.run_oracle(xh, mode))
    _parity.check_rows(xh, mode, dbg, seqs=[0, 37])
