"""specv_verify_noalloc: the entry point for callers that cannot let the
library allocate device memory.  It must give the same outputs as
specv_verify on the same inputs, call after call (its scratch array is reused
and must not leak state from one call into the next).

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import workloads
from tests import _parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    import speculative_decoding_verification_specv_gb300 as specv
    lib = specv.load(build_if_missing=True)
    vp = ctypes.c_void_p
    lib.specv_verify_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int, ctypes.c_int, vp, vp, vp]
    lib.specv_verify_noalloc.restype = ctypes.c_int
    return lib


def _noalloc(lib, x, mode):
    zt = x["target_logits"]
    B, K1, V = zt.shape
    tok = torch.full((B, K1), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    st = lib.specv_verify_noalloc(
        zt.data_ptr(), x["draft_logits"].data_ptr(), x["draft_tokens"].data_ptr(),
        x["u_accept"].data_ptr(), x["u_resample"].data_ptr(), x["lam"].data_ptr(), B, K1 - 1, V,
        1 if zt.dtype == torch.bfloat16 else 0, mode, tok.data_ptr(), n.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return tok, n


@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("cfg", [3, 4])
def test_noalloc_matches_specv_verify_on_two_calls(lib, cfg, mode):
    import speculative_decoding_verification_specv_gb300 as specv
    w = workloads.WORKLOADS[cfg].scaled(B=12)
    for call in range(2):  # two calls in a row, different inputs
        x = workloads.make_inputs(w, DEV, seed_offset=call)
        ref_tok, ref_n = specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                                      x["u_accept"], x["u_resample"], x["lam"], mode=mode)
        tok, n = _noalloc(lib, x, mode)
        torch.cuda.synchronize()
        tok, n = tok.cpu().numpy(), n.cpu().numpy()
        ref_tok, ref_n = ref_tok.cpu().numpy(), ref_n.cpu().numpy()
        # both against the oracle with the tolerance of the parity tests
        xh = _parity.to_host(x)
        orc = _parity.run_oracle(xh, mode)
        _parity.compare(xh, mode, tok, n, orc)
        _parity.compare(xh, mode, ref_tok, ref_n, orc)
        # and against each other outside the decision band
        far = (orc.accept_margin >= _parity.BAND) & (orc.cdf_margin >= _parity.BAND)
        assert (n[far] == ref_n[far]).all() and (tok[far] == ref_tok[far]).all()


@pytest.mark.parametrize("cfg", [3, 4])
def test_noalloc_greedy_matches_specv_verify_exactly(lib, cfg):
    """Greedy verification (an argmax decision, taken in fp32 on both paths):
    the outputs equal specv_verify's exactly, on two calls in a row."""
    import speculative_decoding_verification_specv_gb300 as specv
    w = workloads.WORKLOADS[cfg].scaled(B=12)
    for call in range(2):
        x = workloads.make_inputs(w, DEV, seed_offset=10 + call)
        ref_tok, ref_n = specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                                      x["u_accept"], x["u_resample"], x["lam"], mode=2)
        tok, n = _noalloc(lib, x, 2)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok) and torch.equal(n, ref_n)


@pytest.mark.parametrize("mode", [0, 2], ids=["prob", "greedy"])
def test_noalloc_at_the_array_limit(lib, mode):
    """B*(K+1) = 49152 positions, the most the array holds: the last
    position's statistics end exactly where the counters begin.  Two calls in
    a row, both against the oracle (exact outside the bands)."""
    w = workloads.Workload("noalloc-limit", 6144, 7, 32, "f32", "corr:1.5:0.8:1.0", (0.3,), 31)
    for call in range(2):
        x = workloads.make_inputs(w, DEV, seed_offset=20 + call)
        tok, n = _noalloc(lib, x, mode)
        torch.cuda.synchronize()
        xh = _parity.to_host(x)
        tok, n = tok.cpu().numpy(), n.cpu().numpy()
        if mode == 2:
            import oracle
            orc = oracle.verify_greedy(xh["target_logits"], xh["draft_logits"],
                                       xh["draft_tokens"], xh["lam"])
            _parity.compare_greedy(xh, tok, n, orc)
        else:
            _parity.compare(xh, mode, tok, n, _parity.run_oracle(xh, mode))


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    # B*(K+1) above the array's 49152 positions: refused before any launch
    null = None
    st = lib.specv_verify_noalloc(16, 16, 16, 16, 16, 16, 10000, 8, 32, 0, 0, 16, 16, null)
    assert st == 1
    # one position too many (3781 * 13 = 49153)
    st = lib.specv_verify_noalloc(16, 16, 16, 16, 16, 16, 3781, 12, 32, 0, 0, 16, 16, null)
    assert st == 1
