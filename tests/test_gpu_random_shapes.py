"""GPU parity on seeded random shapes, against the fp64 oracle.

Each case draws a batch size, draft length, vocabulary, logit type, mode,
generator recipe and lambda distribution from one of six families, chosen so
that together they walk every plan the library makes: short aligned rows (the
TMA tile kernel), short misaligned rows (the generic tile kernel), one or two
sequences of long rows (the resident row kernel), one-wave batches of 19-38
sequences (the sequence-cluster kernel), one-wave batches of more sequences
(the streaming kernel with the draws in a second launch) and batches of many
waves (the streaming kernel with early exit).  The decisions must agree with
the oracle bit for bit outside the decision band, and be valid outcomes inside
it (tests/_parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

FAMILIES = ["tile-tma", "tile", "rows-resident", "rows-seq", "rows-stream-split",
            "rows-stream-exit"]
N_CASES = 72


@pytest.fixture(scope="module")
def specv():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    import speculative_decoding_verification_specv_gb300 as m
    m.load(build_if_missing=True)
    return m


def _draw_case(seed):
    """(family, Workload, mode) of case `seed`."""
    rng = np.random.default_rng(7000 + seed)
    fam = FAMILIES[seed % len(FAMILIES)]
    dt = "bf16" if rng.random() < 0.5 else "f32"
    vw = 8 if dt == "bf16" else 4
    if fam == "tile-tma":
        B, K, V = int(rng.integers(1, 3000)), int(rng.integers(1, 9)), vw * int(rng.integers(1, 256 // vw + 1))
    elif fam == "tile":
        B, K = int(rng.integers(1, 500)), int(rng.integers(1, 7))
        V = int(rng.integers(3, 250)) | 1  # odd: rows off 16-byte boundaries
    elif fam == "rows-resident":
        B, K, V = int(rng.integers(1, 3)), int(rng.integers(2, 11)), vw * int(rng.integers(20000, 130000) // vw)
    elif fam == "rows-seq":
        B, K = int(rng.integers(19, 39)), int(rng.integers(1, 9))
        V = int(rng.integers(65536 // (2 if dt == "bf16" else 4), 70000))
    elif fam == "rows-stream-split":
        B, K, V = int(rng.integers(40, 80)), int(rng.integers(2, 6)), int(rng.integers(8000, 40000))
    else:
        B, K, V = int(rng.integers(100, 200)), int(rng.integers(4, 9)), int(rng.integers(8192, 20000))
    structure = ["corr:3.0:0.85:1.0", "half_equal:3.0:0.85:1.0", "rho:3.0:0.5:0.95",
                 "corr:2.0:0.6:1.5"][int(rng.integers(0, 4))]
    lam = [(0.0,), (1.0,), (0.35,), ("uniform", 0.0, 1.0)][int(rng.integers(0, 4))]
    mode = int(rng.integers(0, 3))
    w = workloads.Workload(f"random-{seed}", B, K, V, dt, structure, lam, 40 + seed)
    return fam, w, mode


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shape(specv, seed):
    fam, w, mode = _draw_case(seed)
    plan = specv.plan(w.B, w.K, w.V, 1 if w.dtype == "bf16" else 0, mode)
    x = workloads.make_inputs(w, DEV)
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    tok, n = specv.verify(*args, mode=mode)
    torch.cuda.synchronize()
    tok, n = tok.cpu().numpy(), n.cpu().numpy()
    xh = _parity.to_host(x)
    if mode == specv.GREEDY:
        orc = oracle.verify_greedy(xh["target_logits"], xh["draft_logits"], xh["draft_tokens"],
                                   xh["lam"])
        rep = _parity.compare_greedy(xh, tok, n, orc)
    else:
        rep = _parity.compare(xh, mode, tok, n, _parity.run_oracle(xh, mode))
    print(f"{fam}: B={w.B} K={w.K} V={w.V} {w.dtype} {w.structure} lam={w.lam} mode={mode} "
          f"plan={plan}: {rep}")
