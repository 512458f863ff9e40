"""The C-ABI boundary without a GPU: the library loads, exports every entry
point that include/*.h declares, and rejects bad arguments on the host
(status codes, nothing launched).  No compute call is made here."""
import ctypes
import glob
import os
import re

import pytest

import speculative_decoding_verification_specv_gb300 as specv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return specv.load(build_if_missing=True)


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(specv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_symbols()
    assert "specv_verify" in declared and len(declared) >= 6
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(specv.EXPORTED_SYMBOLS) <= set(declared)


def test_version_and_status_strings(lib):
    assert lib.specv_version() >= 100
    for code, name in [(0, "SPECV_OK"), (1, "SPECV_ERR_INVALID_ARG"), (2, "SPECV_ERR_UNSUPPORTED"),
                       (3, "SPECV_ERR_CUDA"), (4, "SPECV_ERR_NO_MEMORY")]:
        assert specv.status_string(code) == name
    assert specv.status_string(99) == "SPECV_ERR_UNKNOWN"


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _call(B=2, K=3, V=100, dtype=0, mode=0, null=None):
    ptrs = [FAKE] * 8
    if null is not None:
        ptrs[null] = None
    t, d, tok, ua, ur, lam, ot, on = ptrs
    return specv.raw_call("specv_verify", t, d, tok, ua, ur, lam, B, K, V, dtype, mode, ot, on,
                          None)


@pytest.mark.parametrize("null", range(8))
def test_null_pointers_are_rejected(lib, null):
    assert _call(null=null) == 1


@pytest.mark.parametrize("kw", [dict(B=0), dict(B=-5), dict(K=0), dict(K=-1), dict(K=4097),
                                dict(V=0), dict(V=-7), dict(dtype=2), dict(dtype=-1),
                                dict(mode=3), dict(mode=-1), dict(B=1 << 40, K=4000, V=1 << 30)])
def test_bad_sizes_and_enums_are_rejected(lib, kw):
    assert _call(**kw) == 1


def test_debug_entry_point_validates_too(lib):
    st = specv.raw_call("specv_verify_debug", None, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 1, 0, 0,
                        FAKE, FAKE, None, None, None, None)
    assert st == 1


def test_plan_selects_kernels(lib):
    p5 = specv.plan(1_000_000, 4, 32, specv.F32)
    assert p5["kernel"] == "tile-tma" and p5["workspace_bytes"] == 0
    assert specv.plan(5, 3, 33, specv.F32)["kernel"] == "tile"  # rows not on 16-byte boundaries
    p4 = specv.plan(256, 8, 128256, specv.F32)
    assert p4["kernel"] == "rows-stream" and p4["ctas"] == 256 * 9 * p4["cluster"]
    assert p4["workspace_bytes"] >= 256 * 9 * 16 + 256 * 4
    p2 = specv.plan(1, 8, 128256, specv.BF16)
    assert p2["kernel"] == "rows-resident" and p2["cluster"] > 1
    # a slice of one row of 2^24 fp32 logits cannot fit shared memory
    assert specv.plan(2, 2, 1 << 24, specv.F32)["kernel"] == "rows-stream"
    with pytest.raises(specv.SpecvError):
        specv.plan(0, 4, 32)


def test_plan_greedy_mode(lib, monkeypatch):
    """Greedy verification (mode 2) never samples: short aligned rows use the
    TMA tile kernel, everything else the streaming row kernel with the position
    statistics and counters only; the variants that exist for the sampler are
    refused; the debug entry point (probabilities) is refused too."""
    assert specv.plan(1_000_000, 4, 32, specv.F32, specv.GREEDY)["kernel"] == "tile-tma"
    p4 = specv.plan(256, 8, 128256, specv.F32, specv.GREEDY)
    # position candidates, arrival counters and the early-exit words (18 waves of CTAs)
    assert p4["kernel"] == "rows-stream" and p4["workspace_bytes"] == 256 * 9 * 16 + 2 * 256 * 4
    assert p4["early_exit"]
    # short rows off 16-byte boundaries: the streaming row kernel, not the generic tile
    assert specv.plan(5, 3, 33, specv.F32, specv.GREEDY)["kernel"] == "rows-stream"
    monkeypatch.setenv("SPECV_ROWS_VARIANT", "resident")
    with pytest.raises(specv.SpecvError):
        specv.plan(256, 8, 128256, specv.F32, specv.GREEDY)
    monkeypatch.delenv("SPECV_ROWS_VARIANT")
    st = specv.raw_call("specv_verify_debug", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 0, 2,
                        FAKE, FAKE, None, None, None, None)
    assert st == 2


def test_plan_cluster_size_model(lib):
    """Streaming cluster size: the power-of-two rule for many waves (the batched
    workload keeps S = 2), waves x (slice + fixed cost) near one wave (192
    positions: S = 3 fills one wave where S = 4 needs two)."""
    assert specv.plan(256, 8, 128256, specv.F32)["cluster"] == 2
    assert specv.plan(256, 8, 128256, specv.F32, specv.GREEDY)["cluster"] == 2
    p3 = specv.plan(32, 5, 152064, specv.BF16, specv.GREEDY)
    assert p3["kernel"] == "rows-stream" and p3["cluster"] == 3 and p3["ctas"] == 192 * 3
    for B, K, V, dt in [(16, 8, 128256, 0), (64, 4, 32000, 1), (8, 4, 128256, 1), (3, 2, 9000, 0)]:
        S = specv.plan(B, K, V, dt)["cluster"]
        assert 1 <= S <= 16


def test_plan_sequence_clusters(lib, monkeypatch):
    """Sampling grids of about one wave with 19 to 38 sequences (on 152 SMs)
    run one cluster of 16 CTAs per sequence (at least 4 KiB of each row per
    CTA) and need no scratch; SPECV_SAMPLE_SPLIT forces the two-launch
    streaming plan, and greedy verification never uses it."""
    monkeypatch.delenv("SPECV_SAMPLE_SPLIT", raising=False)
    for mode in (specv.PROB_MIX, specv.LOGIT_MIX):
        p3 = specv.plan(32, 5, 152064, specv.BF16, mode)
        assert p3 == {"kernel": "rows-seq", "cluster": 16, "ctas": 512, "workspace_bytes": 0,
                      "early_exit": False, "split_draws": False}
    assert specv.plan(24, 6, 40001, specv.F32)["kernel"] == "rows-seq"     # unaligned rows
    assert specv.plan(38, 3, 65536, specv.BF16)["kernel"] == "rows-seq"    # 16 x 38 CTAs: one wave
    assert specv.plan(40, 3, 65536, specv.BF16)["kernel"] == "rows-stream"  # clusters under 16
    assert specv.plan(150, 2, 16384, specv.BF16)["kernel"] == "rows-stream"
    assert specv.plan(8, 4, 128256, specv.BF16)["kernel"] != "rows-seq"     # too few sequences
    assert specv.plan(256, 8, 128256, specv.F32)["kernel"] == "rows-stream"  # many waves
    assert specv.plan(40, 3, 4096, specv.F32)["kernel"] != "rows-seq"       # short rows
    monkeypatch.setenv("SPECV_SAMPLE_SPLIT", "1")
    p = specv.plan(32, 5, 152064, specv.BF16)
    assert p["kernel"] == "rows-stream" and p["cluster"] == 3 and p["split_draws"]
    monkeypatch.delenv("SPECV_SAMPLE_SPLIT")
    # the edges of the rule on 152 SMs: 2 to 4 CTAs per SM, K + 1 <= 64, >= 4 KiB of a row per CTA
    seq = lambda B, K, V, dt: specv.plan(B, K, V, dt)["kernel"] == "rows-seq"
    assert not seq(18, 5, 152064, specv.BF16) and seq(19, 5, 152064, specv.BF16)
    assert seq(38, 5, 152064, specv.BF16) and not seq(39, 5, 152064, specv.BF16)
    assert seq(19, 63, 32768, specv.BF16) and not seq(19, 64, 32768, specv.BF16)
    assert seq(32, 5, 32768, specv.BF16) and not seq(32, 5, 32760, specv.BF16)
    assert seq(32, 5, 16384, specv.F32) and not seq(32, 5, 16376, specv.F32)


def test_plan_early_exit(lib, monkeypatch):
    """Early exit is planned for the streaming kernels on grids of more than
    two waves (the batched workload), not on one-wave grids (the Qwen-shaped
    batch draws in a second launch) nor for the resident or tile kernels;
    SPECV_EARLY_EXIT=0 turns it off.  It adds one scratch word per sequence."""
    monkeypatch.delenv("SPECV_EARLY_EXIT", raising=False)
    for mode in (specv.PROB_MIX, specv.LOGIT_MIX, specv.GREEDY):
        p4 = specv.plan(256, 8, 128256, specv.F32, mode)
        assert p4["early_exit"] and not p4["split_draws"]
    p3 = specv.plan(32, 5, 152064, specv.BF16, specv.GREEDY)
    assert not p3["early_exit"] and not p3["split_draws"]
    assert not specv.plan(1, 8, 128256, specv.BF16)["early_exit"]       # resident
    assert not specv.plan(1_000_000, 4, 32, specv.F32)["early_exit"]    # TMA tile
    ws_on = specv.plan(256, 8, 128256, specv.F32)["workspace_bytes"]
    monkeypatch.setenv("SPECV_EARLY_EXIT", "0")
    p_off = specv.plan(256, 8, 128256, specv.F32)
    assert not p_off["early_exit"] and ws_on == p_off["workspace_bytes"] + 256 * 4
    monkeypatch.delenv("SPECV_EARLY_EXIT")
    with pytest.raises(specv.SpecvError):
        specv.plan(0, 8, 128256, specv.F32)


def _host_call(B=2, K=3, V=100, dtype=0, mode=0, chunks=0, null=None):
    ptrs = [FAKE] * 8
    if null is not None:
        ptrs[null] = None
    t, d, tok, ua, ur, lam, ot, on = ptrs
    return specv.raw_call("specv_verify_host", t, d, tok, ua, ur, lam, B, K, V, dtype, mode, ot,
                          on, chunks, None)


@pytest.mark.parametrize("kw", [dict(null=0), dict(null=5), dict(null=7), dict(B=0), dict(K=4097),
                                dict(V=-1), dict(dtype=3), dict(mode=3), dict(chunks=-1),
                                dict(chunks=65)])
def test_host_entry_point_validates(lib, kw):
    assert _host_call(**kw) == 1


def test_host_entry_point_refuses_staging_beyond_any_device(lib):
    # 2^20 x 2049 rows of 2^20 fp32 logits: sizes the verify step accepts, but
    # petabytes of staging, refused before anything is allocated or launched
    assert _host_call(B=1 << 20, K=1024, V=1 << 20) == 4


def test_host_binding_checks_tensors():
    import torch
    B, K, V = 3, 2, 50
    x = dict(target_logits=torch.zeros(B, K + 1, V), draft_logits=torch.zeros(B, K, V),
             draft_tokens=torch.zeros(B, K, dtype=torch.int32),
             u_accept=torch.zeros(B, K), u_resample=torch.zeros(B), lam=torch.zeros(B))
    outs = dict(out_tokens=torch.empty(B, K + 1, dtype=torch.int32),
                out_n_accepted=torch.empty(B, dtype=torch.int32))
    with pytest.raises(ValueError):
        specv.verify_host(*x.values(), chunks=65, **outs)
    bad = dict(x, draft_tokens=torch.zeros(B, K, dtype=torch.int64))
    with pytest.raises(TypeError):
        specv.verify_host(*bad.values(), **outs)
    with pytest.raises(ValueError):  # CUDA-side entry point on host tensors
        specv.verify(*x.values())


def test_random_shape_families_reach_their_plans(lib):
    """The families of the random-shape GPU parity cases are what they say:
    every family is planned as named at least once (greedy shapes of the
    sampling-only plans go to the streaming kernel)."""
    from tests.test_gpu_random_shapes import FAMILIES, N_CASES, _draw_case
    seen = set()
    for seed in range(N_CASES):
        fam, w, mode = _draw_case(seed)
        p = specv.plan(w.B, w.K, w.V, specv.BF16 if w.dtype == "bf16" else specv.F32, mode)
        name = p["kernel"]
        if name == "rows-stream":
            name = ("rows-stream-split" if p["split_draws"] else
                    "rows-stream-exit" if p["early_exit"] else "rows-stream")
        if name == fam:
            seen.add(fam)
    assert seen == set(FAMILIES), sorted(set(FAMILIES) - seen)
