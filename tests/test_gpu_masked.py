"""GPU parity with masked logits (-inf entries: a padded vocabulary, a grammar
or top-k mask) against the fp64 oracle.

Reading of the pages for masks, in both the kernels and the oracle: in the
logit mixture (1 - lambda) z_t + lambda z_q a -inf entry of positive weight
gives -inf and a term of weight zero drops out (lambda = 0 gives z_t, lambda = 1
gives z_q); a drafted token that the draft row masks has q(x) = 0, so its ratio
is +inf (accepted) unless p~(x) = 0 too (rejected).  Rows here carry random
masked entries, a masked prefix (whole first batches of a thread masked) and
a masked tail (a padded vocabulary), on every kernel family and at lambda in
{0, 0.5, 1}.
"""
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


def _mask(x, seed, prefix, tail):
    """Random 10% of the target and draft entries, a masked prefix and tail of
    every row (both rows), and the drafted token of every third sequence's
    first position moved onto an entry its draft row masks."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    zt, zq = x["target_logits"], x["draft_logits"]
    B, K1, V = zt.shape
    ninf = float("-inf")
    mt = (torch.rand((B, K1, V), generator=g) < 0.1).to(DEV)
    mq = (torch.rand((B, K1 - 1, V), generator=g) < 0.1).to(DEV)
    zt.masked_fill_(mt, ninf)
    zq.masked_fill_(mq, ninf)
    if prefix:
        zt[..., :prefix] = ninf
        zq[..., :prefix] = ninf
    if tail:
        zt[..., V - tail:] = ninf
        zq[..., V - tail:] = ninf
    # some drafted tokens sit on entries the draft row masks (q(x) = 0); keep
    # every row with at least one unmasked entry of each kind
    tok = x["draft_tokens"]
    for b in range(0, B, 3):
        cand = torch.nonzero(zq[b, 0] == ninf).flatten()
        if cand.numel():
            tok[b, 0] = cand[int(torch.randint(cand.numel(), (1,), generator=g))].to(torch.int32)
    return x


SHAPES = [
    # (B, K, V, dtype, prefix, tail): streaming (several waves and one), resident, tile kernels
    (200, 6, 8192, "f32", 2048, 100),     # several waves: draws at the rejection, early exit
    (6, 4, 128256, "f32", 4096, 256),     # one wave: split draws
    (1, 8, 128256, "bf16", 4096, 256),    # resident kernel
    (3000, 4, 32, "f32", 8, 4),           # TMA tile kernel
    (7, 3, 33, "f32", 4, 3),              # generic tile kernel (rows off 16-byte boundaries)
    (4, 3, 4099, "bf16", 512, 17),        # streaming kernel, rows off 16-byte boundaries
]


@pytest.mark.parametrize("lam", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("mode", [0, 1], ids=["prob", "logit"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}")
def test_masked_logits_match_the_oracle(specv, shape, mode, lam):
    B, K, V, dt, prefix, tail = shape
    w = workloads.Workload("masked", B, K, V, dt, "corr:3.0:0.85:1.0", (lam,), 51)
    x = _mask(workloads.make_inputs(w, DEV), seed=V + K, prefix=prefix, tail=tail)
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    tok, n = specv.verify(*args, mode=mode)
    dbg = specv.verify_debug(*args, mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(dbg["tokens"], tok) and torch.equal(dbg["n_accepted"], n)
    tok, n = tok.cpu().numpy(), n.cpu().numpy()
    assert (n >= 0).all()
    xh = _parity.to_host(x)
    orc = _parity.run_oracle(xh, mode)
    rep = _parity.compare(xh, mode, tok, n, orc)
    rep.update(_parity.check_probabilities(xh, mode, dbg, orc))
    rep.update(_parity.check_rows(xh, mode, dbg, seqs=[0, B - 1]))
    # no masked entry is ever emitted where p~ (or the residual) gives it no mass
    for b in range(min(B, 64)):
        t = tok[b, n[b]]
        assert 0 <= t < V
    print(f"{shape} mode={mode} lam={lam}: {rep}")


@pytest.mark.parametrize("lam", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}K{s[1]}V{s[2]}{s[3]}")
def test_masked_logits_greedy(specv, shape, lam):
    B, K, V, dt, prefix, tail = shape
    w = workloads.Workload("masked", B, K, V, dt, "corr:3.0:0.85:1.0", (lam,), 52)
    x = _mask(workloads.make_inputs(w, DEV), seed=V + 7, prefix=prefix, tail=tail)
    tok, n = specv.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                          x["u_accept"], x["u_resample"], x["lam"], mode=specv.GREEDY)
    torch.cuda.synchronize()
    xh = _parity.to_host(x)
    orc = oracle.verify_greedy(xh["target_logits"], xh["draft_logits"], xh["draft_tokens"],
                               xh["lam"])
    rep = _parity.compare_greedy(xh, tok.cpu().numpy(), n.cpu().numpy(), orc)
    print(f"greedy {shape} lam={lam}: {rep}")
