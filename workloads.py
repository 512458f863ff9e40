"""Seeded synthetic inputs for the verify/accept step.

This module is shared by the tests, the smoke check and the benchmark.  It
feeds both the CUDA library and the CPU oracle with the same bytes, and holds
none of the method's arithmetic (no softmax, mixture, acceptance test or
inverse CDF): draft tokens are drawn by the Gumbel-max trick, which samples
exactly from softmax(draft logits) without forming that softmax.

The five workloads stand in for the pages' long-context workloads
(Llama-3.1 and Qwen2.5 targets on a long-context evaluation suite); only the
vocabulary sizes of those model families are borrowed.  Logits are Gaussian
with the stated scales and draft/target correlation; bf16 logits are rounded
from fp32 by round-to-nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

SEED_BASE = 20260


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    V: int
    dtype: str            # "f32" or "bf16"
    structure: str        # generator recipe, see make_inputs
    lam: tuple            # lambda (scalar) or ("uniform", lo, hi) per sequence
    index: int            # 1-based workload number (seed offset)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def roofline_bytes(self) -> int:
        """Every logit read once: (2K+1)*B*V*sizeof(dtype)."""
        return (2 * self.K + 1) * self.B * self.V * self.elem_bytes

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    1: Workload("tiny-v1000-f32", 1, 4, 1000, "f32", "corr:2.0:0.8:1.0", (0.3,), 1),
    2: Workload("llama3-v128256-bf16-b1", 1, 8, 128256, "bf16", "corr:3.0:0.9:0.7", (0.5,), 2),
    3: Workload("qwen25-v152064-bf16-b32", 32, 5, 152064, "bf16", "rho:3.0:0.5:0.95",
                ("uniform", 0.0, 0.5), 3),
    4: Workload("batched-v128256-f32-b256", 256, 8, 128256, "f32", "half_equal:3.0:0.85:1.0",
                (0.2,), 4),
    5: Workload("exactness-v32-f32-b1e6", 1_000_000, 4, 32, "f32", "broadcast:1.5", (0.25,), 5),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _gumbel_max_tokens(zq32: torch.Tensor, g, device) -> torch.Tensor:
    """argmax_v (z_v + G_v) with G_v standard Gumbel: a draw from softmax(z)."""
    B, K, V = zq32.shape
    out = torch.empty((B, K), dtype=torch.int32, device=device)
    # chunk over sequences to bound the temporary
    step = max(1, (1 << 27) // max(1, K * V))
    for b0 in range(0, B, step):
        b1 = min(B, b0 + step)
        u = torch.rand((b1 - b0, K, V), generator=g, device=device, dtype=torch.float32)
        u.clamp_(min=torch.finfo(torch.float32).tiny)
        gum = -torch.log(-torch.log(u))
        out[b0:b1] = torch.argmax(zq32[b0:b1] + gum, dim=-1).to(torch.int32)
    return out


def make_inputs(w: Workload, device="cpu", seed_offset: int = 0, lam=None):
    """Seeded inputs of workload ``w`` on ``device``.

    Returns a dict of tensors: target_logits [B][K+1][V], draft_logits [B][K][V]
    (dtype of the workload), draft_tokens int32 [B][K], u_accept fp32 [B][K],
    u_resample fp32 [B], lam fp32 [B].  ``lam`` overrides the workload's
    lambda with a scalar.

    Recipes (``structure``):
      corr:s:a:e        z_t ~ N(0, s^2); z_q = a*z_t + N(0, e^2)
      rho:s:lo:hi       z_t ~ N(0, s^2); per sequence rho ~ U(lo, hi);
                        z_q = rho*z_t + sqrt(1 - rho^2)*s*eps (equal marginal variance)
      half_equal:s:a:e  as corr for sequences b < B/2; z_q = z_t[:, :K] for b >= B/2
      broadcast:s       one z_t [K+1][V] and one independent z_q [K][V], both
                        N(0, s^2), copied to every sequence (independent trials)
    """
    device = torch.device(device)
    base = (SEED_BASE + w.index) * 100 + seed_offset * 10
    g_t, g_q, g_tok, g_u, g_lam = (_gen(device, base + k) for k in range(5))
    B, K, V = w.B, w.K, w.V
    kind, *params = w.structure.split(":")
    p = [float(x) for x in params]
    if kind == "corr":
        s, a, e = p
        zt = _randn((B, K + 1, V), g_t, device).mul_(s)
        zq = zt[:, :K].mul(a).add_(_randn((B, K, V), g_q, device).mul_(e))
    elif kind == "rho":
        s, lo, hi = p
        zt = _randn((B, K + 1, V), g_t, device).mul_(s)
        rho = torch.rand((B, 1, 1), generator=g_q, device=device) * (hi - lo) + lo
        eps = _randn((B, K, V), g_q, device)
        zq = zt[:, :K] * rho + torch.sqrt(1.0 - rho * rho) * s * eps
    elif kind == "half_equal":
        s, a, e = p
        zt = _randn((B, K + 1, V), g_t, device).mul_(s)
        zq = zt[:, :K].mul(a).add_(_randn((B, K, V), g_q, device).mul_(e))
        h = B // 2
        zq[h:] = zt[h:, :K]
    elif kind == "broadcast":
        (s,) = p
        zt1 = _randn((1, K + 1, V), g_t, device).mul_(s)
        zq1 = _randn((1, K, V), g_q, device).mul_(s)
        zt = zt1.expand(B, K + 1, V).contiguous()
        zq = zq1.expand(B, K, V).contiguous()
    else:
        raise ValueError(f"unknown structure {w.structure}")
    zt = zt.to(w.torch_dtype).contiguous()
    zq = zq.to(w.torch_dtype).contiguous()
    tokens = _gumbel_max_tokens(zq.float(), g_tok, device)
    u_accept = torch.rand((B, K), generator=g_u, device=device, dtype=torch.float32)
    u_resample = torch.rand((B,), generator=g_u, device=device, dtype=torch.float32)
    if lam is not None:
        lam_t = torch.full((B,), float(lam), dtype=torch.float32, device=device)
    elif w.lam[0] == "uniform":
        _, lo, hi = w.lam
        lam_t = torch.rand((B,), generator=g_lam, device=device) * (hi - lo) + lo
    else:
        lam_t = torch.full((B,), float(w.lam[0]), dtype=torch.float32, device=device)
    return dict(target_logits=zt, draft_logits=zq, draft_tokens=tokens, u_accept=u_accept,
                u_resample=u_resample, lam=lam_t.to(torch.float32).contiguous())


def tree_shape(kind: str, N: int, seed: int = 0):
    """Parent list [N+1] (-1 at the root, parent[j] < j) of a draft tree.
      chain      parent[j] = j - 1
      kary:k     breadth-first k-ary tree (each node's children contiguous)
      star       every node a child of the root
      random:f   parent[j] uniform in [max(0, j - f), j)
    """
    name, *rest = kind.split(":")
    par = [-1]
    if name == "chain":
        par += [j - 1 for j in range(1, N + 1)]
    elif name == "kary":
        k = int(rest[0])
        par += [(j - 1) // k for j in range(1, N + 1)]
    elif name == "star":
        par += [0] * N
    elif name == "random":
        f = int(rest[0])
        g = torch.Generator().manual_seed(SEED_BASE * 7 + seed)
        for j in range(1, N + 1):
            lo = max(0, j - f)
            par.append(lo + int(torch.randint(0, j - lo, (1,), generator=g)))
    else:
        raise ValueError(f"unknown tree shape {kind}")
    return par


def make_tree_inputs(B: int, N: int, V: int, dtype: str = "f32", shape: str = "kary:2",
                     s: float = 3.0, a: float = 0.8, e: float = 1.0, lam: float = 0.3,
                     seed: int = 0, device="cpu"):
    """Seeded inputs of tree verification: the same tree for every sequence.

    Every node u has a target row z_t[u] ~ N(0, s^2); every node with children
    has a draft row z_q = a * z_t[u] + N(0, e^2), numbered in node order; the
    children of u are drawn independently from softmax(z_q) by the Gumbel-max
    trick (the tree verification reading: siblings are i.i.d. draft samples).
    Returns target_logits [B][N+1][V], draft_logits [B][M][V], parent,
    draft_row, tokens (int32 [B][N+1]), u_accept [B][N+1], u_resample [B], lam
    [B].
    """
    device = torch.device(device)
    par = tree_shape(shape, N, seed)
    has_child = [False] * (N + 1)
    for j in range(1, N + 1):
        has_child[par[j]] = True
    drow = []
    M = 0
    for u in range(N + 1):
        drow.append(M if has_child[u] else -1)
        M += 1 if has_child[u] else 0
    base = (SEED_BASE + 50 + seed) * 100
    g_t, g_q, g_tok, g_u = (_gen(device, base + k) for k in range(4))
    torch_dtype = torch.bfloat16 if dtype == "bf16" else torch.float32
    zt = _randn((B, N + 1, V), g_t, device).mul_(s)
    rows_of = [u for u in range(N + 1) if has_child[u]]
    zq = torch.empty((B, M, V), dtype=torch.float32, device=device)
    if M:
        zq.copy_(zt[:, rows_of].mul(a).add_(_randn((B, M, V), g_q, device).mul_(e)))
    zt = zt.to(torch_dtype).contiguous()
    zq = zq.to(torch_dtype).contiguous()
    tokens = torch.zeros((B, N + 1), dtype=torch.int32, device=device)
    if N:
        child_rows = torch.tensor([drow[par[j]] for j in range(1, N + 1)], device=device)
        zq_children = zq.float().index_select(1, child_rows)  # [B][N][V]: parent's draft row
        tokens[:, 1:] = _gumbel_max_tokens(zq_children, g_tok, device)
    u_accept = torch.rand((B, N + 1), generator=g_u, device=device, dtype=torch.float32)
    u_resample = torch.rand((B,), generator=g_u, device=device, dtype=torch.float32)
    parent_t = torch.tensor(par, dtype=torch.int32, device=device).repeat(B, 1).contiguous()
    drow_t = torch.tensor(drow, dtype=torch.int32, device=device).repeat(B, 1).contiguous()
    return dict(target_logits=zt, draft_logits=zq, parent=parent_t, draft_row=drow_t,
                tokens=tokens, u_accept=u_accept, u_resample=u_resample,
                lam=torch.full((B,), float(lam), dtype=torch.float32, device=device))


def expected_bytes(w: Workload) -> int:
    return w.roofline_bytes


def describe(w: Workload) -> str:
    return (f"{w.name}: B={w.B} K={w.K} V={w.V} {w.dtype} {w.structure} lambda={w.lam}; "
            f"roofline bytes={w.roofline_bytes} ({w.roofline_bytes / 2**20:.1f} MiB)")


if __name__ == "__main__":  # pragma: no cover
    for k, w in WORKLOADS.items():
        print(k, describe(w), f"{math.log2(max(1, w.V)):.1f} bits/token")
