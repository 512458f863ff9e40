"""GB300-native speculative-decoding verify/accept with RAPID knowledge transfer.

A thin ctypes binding over ``libspecv.so`` (C ABI in ``include/specv.h``).
Every step of the verify path runs in the library's CUDA kernels; this module
only checks tensor metadata, passes device pointers and the current CUDA
stream, and turns status codes into exceptions.  PyTorch provides device
memory and streams.  There is no CPU fallback: if the library is missing the
calls raise.

Sources (page title, section): "RAPID：基于检索增强的推测解码长上下文推理",
"2) 推理时知识迁移" (p~ = (1-λ) p_t + λ p_q) and "3) 候选验证机制（伪代码）"
(the per-step acceptance loop); "大模型推理的Speculative Decoding原理详解",
"修改的拒绝采样"; "投机解码（EAGLE）…", "1. 为什么无损" (resample from
max(0, p - q)).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = ["SpecvError", "PROB_MIX", "LOGIT_MIX", "GREEDY", "F32", "BF16", "load", "lib_path",
           "verify", "verify_host", "verify_debug", "verify_tree", "acceptance_rates", "choose_k",
           "AdaptiveK", "plan", "status_string", "EXPORTED_SYMBOLS"]

PROB_MIX = 0
LOGIT_MIX = 1
GREEDY = 2
F32 = 0
BF16 = 1

EXPORTED_SYMBOLS = ("specv_verify", "specv_verify_debug", "specv_plan", "specv_status_string",
                    "specv_last_cuda_error", "specv_version", "specv_verify_noalloc",
                    "specv_acceptance_rates", "specv_choose_k", "specv_verify_tree",
                    "specv_verify_host")

_STATUS = {0: "SPECV_OK", 1: "SPECV_ERR_INVALID_ARG", 2: "SPECV_ERR_UNSUPPORTED",
           3: "SPECV_ERR_CUDA", 4: "SPECV_ERR_NO_MEMORY"}


class SpecvError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what}: {_STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libspecv.so (optionally building it first).  Raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            _build.build()
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(
                f"libspecv.so not found at {_build.LIB_PATH}; build it with "
                "`python -m speculative_decoding_verification_specv_gb300.build`")
        lib = ctypes.CDLL(_build.LIB_PATH)
        vp, i32p, f32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int32
        common = [vp, vp, vp, vp, vp, vp, i64, i32, i32, ctypes.c_int, ctypes.c_int, vp, vp]
        lib.specv_verify.argtypes = common + [vp]
        lib.specv_verify.restype = ctypes.c_int
        lib.specv_verify_host.argtypes = common + [i32, vp]
        lib.specv_verify_host.restype = ctypes.c_int
        lib.specv_verify_debug.argtypes = common + [vp, vp, vp, vp]
        lib.specv_verify_debug.restype = ctypes.c_int
        lib.specv_plan.argtypes = [i64, i32, i32, ctypes.c_int, ctypes.c_int, i32p, i32p,
                                   ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.specv_plan.restype = ctypes.c_int
        lib.specv_plan_flags.argtypes = [i64, i32, i32, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_uint32)]
        lib.specv_plan_flags.restype = ctypes.c_int
        lib.specv_status_string.argtypes = [ctypes.c_int]
        lib.specv_status_string.restype = ctypes.c_char_p
        lib.specv_last_cuda_error.argtypes = []
        lib.specv_last_cuda_error.restype = ctypes.c_char_p
        lib.specv_version.argtypes = []
        lib.specv_version.restype = ctypes.c_int32
        lib.specv_acceptance_rates.argtypes = [vp, vp, vp, i64, i32, i32, ctypes.c_int,
                                               ctypes.c_int, vp, vp]
        lib.specv_acceptance_rates.restype = ctypes.c_int
        lib.specv_verify_tree.argtypes = [vp] * 8 + [i64, i32, i32, i32, ctypes.c_int,
                                                     ctypes.c_int, vp, vp, vp, vp]
        lib.specv_verify_tree.restype = ctypes.c_int
        lib.specv_verify_host_direct.argtypes = common + [vp]
        lib.specv_verify_host_direct.restype = ctypes.c_int
        lib.specv_verify_host_early_exit.argtypes = common + [ctypes.POINTER(i64),
                                                              ctypes.POINTER(i64), vp]
        lib.specv_verify_host_early_exit.restype = ctypes.c_int
        lib.specv_release_stream.argtypes = [vp]
        lib.specv_release_stream.restype = ctypes.c_int
        lib.specv_shard_bounds.argtypes = [i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.specv_shard_bounds.restype = ctypes.c_int
        lib.specv_verify_sharded_host.argtypes = common + [i32, vp]
        lib.specv_verify_sharded_host.restype = ctypes.c_int
        dbl = ctypes.c_double
        lib.specv_choose_k.argtypes = [dbl, dbl, dbl, dbl, i32, i32]
        lib.specv_choose_k.restype = ctypes.c_int32
        _ = f32p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().specv_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        detail = load().specv_last_cuda_error().decode() if status == 3 else ""
        raise SpecvError(status, what, detail)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _require(t: torch.Tensor, name: str, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _args(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lam, mode, out_tokens,
          out_n_accepted, host=False):
    zt, zq = target_logits, draft_logits
    if zt.dim() != 3:
        raise ValueError("target_logits must be [B][K+1][V]")
    B, K1, V = zt.shape
    K = K1 - 1
    dev = zt.device
    if host and dev.type != "cpu":
        raise ValueError("verify_host takes tensors in host memory (use verify for CUDA tensors)")
    if not host and dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors (the verify step runs only on the GPU)")
    _require(zt, "target_logits", None, (B, K + 1, V), dev)
    _require(zq, "draft_logits", zt.dtype, (B, K, V), dev)
    _require(draft_tokens, "draft_tokens", torch.int32, (B, K), dev)
    _require(u_accept, "u_accept", torch.float32, (B, K), dev)
    _require(u_resample, "u_resample", torch.float32, (B,), dev)
    _require(lam, "lam", torch.float32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev, pin_memory=host)
    if out_n_accepted is None:
        out_n_accepted = torch.empty((B,), dtype=torch.int32, device=dev, pin_memory=host)
    _require(out_tokens, "out_tokens", torch.int32, (B, K + 1), dev)
    _require(out_n_accepted, "out_n_accepted", torch.int32, (B,), dev)
    if mode not in (PROB_MIX, LOGIT_MIX, GREEDY):
        raise ValueError("mode must be PROB_MIX (0), LOGIT_MIX (1) or GREEDY (2)")
    return B, K, V, dev, out_tokens, out_n_accepted


def _stream_ptr(stream, dev):
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return ctypes.c_void_p(s.cuda_stream)


def verify(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lam,
           mode: int = PROB_MIX, out_tokens=None, out_n_accepted=None, stream=None):
    """One verify/accept step on the GPU.  Returns (out_tokens [B][K+1], out_n [B]).

    mode: PROB_MIX or LOGIT_MIX (the sampling rule with the mixture p~), or
    GREEDY (accept x_i iff it is the argmax of the mixed logits of row i; the
    uniforms are not read).

    All tensors are CUDA, contiguous: target_logits [B][K+1][V] and
    draft_logits [B][K][V] (float32 or bfloat16), draft_tokens int32 [B][K],
    u_accept float32 [B][K], u_resample float32 [B], lam float32 [B].  Runs
    asynchronously on ``stream`` (default: the current stream).
    """
    B, K, V, dev, out_tokens, out_n = _args(target_logits, draft_logits, draft_tokens, u_accept,
                                            u_resample, lam, mode, out_tokens, out_n_accepted)
    st = load().specv_verify(
        target_logits.data_ptr(), draft_logits.data_ptr(), draft_tokens.data_ptr(),
        u_accept.data_ptr(), u_resample.data_ptr(), lam.data_ptr(), B, K, V,
        _dtype_code(target_logits), int(mode), out_tokens.data_ptr(), out_n.data_ptr(),
        _stream_ptr(stream, dev))
    _check(st, "specv_verify")
    return out_tokens, out_n


def verify_host(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lam,
                mode: int = PROB_MIX, out_tokens=None, out_n_accepted=None, chunks: int = 0,
                stream=None):
    """verify() on tensors in host memory (page-locked for asynchronous copies):
    the library copies the inputs to the GPU in chunks of whole sequences,
    overlapping each chunk's copy with the verify step of the previous one, and
    copies the results back into out_tokens / out_n_accepted (host tensors,
    page-locked ones allocated if not given).  Asynchronous on ``stream``
    (default: the current stream of the current device): synchronise it before
    reading the outputs or changing the inputs.  chunks: 0 = the library's
    choice, else 1..64."""
    B, K, V, _, out_tokens, out_n = _args(target_logits, draft_logits, draft_tokens, u_accept,
                                          u_resample, lam, mode, out_tokens, out_n_accepted,
                                          host=True)
    if not 0 <= int(chunks) <= 64:
        raise ValueError("chunks must be in 0..64")
    dev = stream.device if stream is not None else torch.device("cuda",
                                                                torch.cuda.current_device())
    st = load().specv_verify_host(
        target_logits.data_ptr(), draft_logits.data_ptr(), draft_tokens.data_ptr(),
        u_accept.data_ptr(), u_resample.data_ptr(), lam.data_ptr(), B, K, V,
        _dtype_code(target_logits), int(mode), out_tokens.data_ptr(), out_n.data_ptr(),
        int(chunks), _stream_ptr(stream, dev))
    _check(st, "specv_verify_host")
    return out_tokens, out_n


def verify_host_direct(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lam,
                       mode: int = PROB_MIX, out_tokens=None, out_n_accepted=None, stream=None):
    """verify() on host tensors that the GPU reads and writes in place (page-locked,
    e.g. ``pin_memory()``): the kernels load only the rows they reach over the host
    link.  Asynchronous on ``stream``; the outputs (page-locked ones allocated if
    not given) are complete once it has completed."""
    B, K, V, _, out_tokens, out_n = _args(target_logits, draft_logits, draft_tokens, u_accept,
                                          u_resample, lam, mode, out_tokens, out_n_accepted,
                                          host=True)
    dev = stream.device if stream is not None else torch.device("cuda",
                                                                torch.cuda.current_device())
    st = load().specv_verify_host_direct(
        target_logits.data_ptr(), draft_logits.data_ptr(), draft_tokens.data_ptr(),
        u_accept.data_ptr(), u_resample.data_ptr(), lam.data_ptr(), B, K, V,
        _dtype_code(target_logits), int(mode), out_tokens.data_ptr(), out_n.data_ptr(),
        _stream_ptr(stream, dev))
    _check(st, "specv_verify_host_direct")
    return out_tokens, out_n


def verify_host_early_exit(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lam,
                           mode: int = PROB_MIX, out_tokens=None, out_n_accepted=None,
                           stream=None):
    """verify_host() that copies only the rows the verify step reaches, position
    by position (a small read-back of the live sequences per position).  Returns
    (out_tokens, out_n, h2d_bytes, d2h_bytes): the outputs are complete once
    ``stream`` has completed; the byte counts are what crossed the host link."""
    B, K, V, _, out_tokens, out_n = _args(target_logits, draft_logits, draft_tokens, u_accept,
                                          u_resample, lam, mode, out_tokens, out_n_accepted,
                                          host=True)
    dev = stream.device if stream is not None else torch.device("cuda",
                                                                torch.cuda.current_device())
    h2d, d2h = ctypes.c_int64(0), ctypes.c_int64(0)
    st = load().specv_verify_host_early_exit(
        target_logits.data_ptr(), draft_logits.data_ptr(), draft_tokens.data_ptr(),
        u_accept.data_ptr(), u_resample.data_ptr(), lam.data_ptr(), B, K, V,
        _dtype_code(target_logits), int(mode), out_tokens.data_ptr(), out_n.data_ptr(),
        ctypes.byref(h2d), ctypes.byref(d2h), _stream_ptr(stream, dev))
    _check(st, "specv_verify_host_early_exit")
    return out_tokens, out_n, h2d.value, d2h.value


def release_stream(stream=None):
    """Free the scratch and staging the library keeps for ``stream`` (default:
    the current stream) on the current device, after the stream's queued work;
    only once no CUDA graph captured from library calls on it will be replayed."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(load().specv_release_stream(_stream_ptr(stream, dev)), "specv_release_stream")


def shard_bounds(B: int, n_shards: int, shard: int) -> tuple[int, int]:
    """Sequences [lo, hi) of shard `shard` of a batch of B split over n_shards
    (the library's split: contiguous, in order, sizes within one)."""
    lo, hi = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(load().specv_shard_bounds(int(B), int(n_shards), int(shard), ctypes.byref(lo),
                                     ctypes.byref(hi)), "specv_shard_bounds")
    return lo.value, hi.value


def verify_sharded(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lam,
                   devices, mode: int = PROB_MIX, out_tokens=None, out_n_accepted=None):
    """One batch in host memory verified on several devices: shard g of
    len(devices) (shard_bounds) runs on CUDA device devices[g], and its outputs
    land at its offset in out_tokens / out_n_accepted (host tensors, page-locked
    ones allocated if not given).  Synchronous: returns the outputs complete."""
    B, K, V, _, out_tokens, out_n = _args(target_logits, draft_logits, draft_tokens, u_accept,
                                          u_resample, lam, mode, out_tokens, out_n_accepted,
                                          host=True)
    devs = (ctypes.c_int32 * len(devices))(*[int(d) for d in devices])
    st = load().specv_verify_sharded_host(
        target_logits.data_ptr(), draft_logits.data_ptr(), draft_tokens.data_ptr(),
        u_accept.data_ptr(), u_resample.data_ptr(), lam.data_ptr(), B, K, V,
        _dtype_code(target_logits), int(mode), out_tokens.data_ptr(), out_n.data_ptr(),
        len(devices), devs)
    _check(st, "specv_verify_sharded_host")
    return out_tokens, out_n


def verify_debug(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lam,
                 mode: int = PROB_MIX, stream=None):
    """verify() plus p~(x_i), q(x_i) [B][K] and the row log-normalisers [B][K+1][2]."""
    B, K, V, dev, out_tokens, out_n = _args(target_logits, draft_logits, draft_tokens, u_accept,
                                            u_resample, lam, mode, None, None)
    px = torch.full((B, K), float("nan"), dtype=torch.float32, device=dev)
    qx = torch.full((B, K), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((B, K + 1, 2), float("nan"), dtype=torch.float32, device=dev)
    st = load().specv_verify_debug(
        target_logits.data_ptr(), draft_logits.data_ptr(), draft_tokens.data_ptr(),
        u_accept.data_ptr(), u_resample.data_ptr(), lam.data_ptr(), B, K, V,
        _dtype_code(target_logits), int(mode), out_tokens.data_ptr(), out_n.data_ptr(),
        px.data_ptr(), qx.data_ptr(), lse.data_ptr(), _stream_ptr(stream, dev))
    _check(st, "specv_verify_debug")
    return dict(tokens=out_tokens, n_accepted=out_n, ptilde_x=px, q_x=qx, lse=lse)


def verify_tree(target_logits, draft_logits, parent, draft_row, tokens, u_accept, u_resample,
                lam, mode: int = PROB_MIX, stream=None):
    """Tree verification on the GPU.  target_logits [B][N+1][V], draft_logits
    [B][M][V] (same dtype; M may be 0), parent/draft_row/tokens int32 [B][N+1],
    u_accept float32 [B][N+1], u_resample and lam float32 [B].  Returns
    (out_tokens [B][N+1], out_path [B][N+1], out_n [B])."""
    zt, zq = target_logits, draft_logits
    if zt.dim() != 3 or zq.dim() != 3:
        raise ValueError("target_logits must be [B][N+1][V] and draft_logits [B][M][V]")
    B, N1, V = zt.shape
    M = zq.shape[1]
    dev = zt.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors (the verify step runs only on the GPU)")
    _require(zt, "target_logits", None, (B, N1, V), dev)
    _require(zq, "draft_logits", zt.dtype, (B, M, V), dev)
    for name, t in (("parent", parent), ("draft_row", draft_row), ("tokens", tokens)):
        _require(t, name, torch.int32, (B, N1), dev)
    _require(u_accept, "u_accept", torch.float32, (B, N1), dev)
    _require(u_resample, "u_resample", torch.float32, (B,), dev)
    _require(lam, "lam", torch.float32, (B,), dev)
    if mode not in (PROB_MIX, LOGIT_MIX):
        raise ValueError("mode must be PROB_MIX (0) or LOGIT_MIX (1)")
    out_tokens = torch.empty((B, N1), dtype=torch.int32, device=dev)
    out_path = torch.empty((B, N1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    st = load().specv_verify_tree(
        zt.data_ptr(), zq.data_ptr() if M > 0 else None, parent.data_ptr(), draft_row.data_ptr(),
        tokens.data_ptr(), u_accept.data_ptr(), u_resample.data_ptr(), lam.data_ptr(), B, N1 - 1,
        M, V, _dtype_code(zt), int(mode), out_tokens.data_ptr(), out_path.data_ptr(),
        out_n.data_ptr(), _stream_ptr(stream, dev))
    _check(st, "specv_verify_tree")
    return out_tokens, out_path, out_n


def acceptance_rates(target_logits, draft_logits, lam, mode: int = PROB_MIX, out=None,
                     stream=None):
    """Exact acceptance probability alpha [B][K] = sum_v min(p~_v, q_v) of every
    drafted position (float32, on the logits' device; NaN where lam is outside
    [0, 1]).  Same tensor rules as verify(); mode PROB_MIX or LOGIT_MIX."""
    zt, zq = target_logits, draft_logits
    if zt.dim() != 3:
        raise ValueError("target_logits must be [B][K+1][V]")
    B, K1, V = zt.shape
    K = K1 - 1
    dev = zt.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors (the kernels run only on the GPU)")
    _require(zt, "target_logits", None, (B, K + 1, V), dev)
    _require(zq, "draft_logits", zt.dtype, (B, K, V), dev)
    _require(lam, "lam", torch.float32, (B,), dev)
    if mode not in (PROB_MIX, LOGIT_MIX):
        raise ValueError("mode must be PROB_MIX (0) or LOGIT_MIX (1)")
    if out is None:
        out = torch.empty((B, K), dtype=torch.float32, device=dev)
    _require(out, "out", torch.float32, (B, K), dev)
    st = load().specv_acceptance_rates(zt.data_ptr(), zq.data_ptr(), lam.data_ptr(), B, K, V,
                                       _dtype_code(zt), int(mode), out.data_ptr(),
                                       _stream_ptr(stream, dev))
    _check(st, "specv_acceptance_rates")
    return out


def choose_k(alpha: float, cost_draft: float, cost_verify_fixed: float,
             cost_verify_per_token: float = 0.0, k_min: int = 1, k_max: int = 16) -> int:
    """Draft length maximising (1 + a + ... + a^K) / (fixed + K (draft + per-token))."""
    k = load().specv_choose_k(float(alpha), float(cost_draft), float(cost_verify_fixed),
                              float(cost_verify_per_token), int(k_min), int(k_max))
    if k < 0:
        raise ValueError("specv_choose_k: alpha must be in [0, 1], costs >= 0 with a positive "
                         "step cost, and 1 <= k_min <= k_max <= 4096")
    return int(k)


class AdaptiveK:
    """Host-side draft-length controller: a running mean of the acceptance
    probabilities of recent steps (from acceptance_rates, or any estimate)
    and the K that specv_choose_k picks for it."""

    def __init__(self, cost_draft: float, cost_verify_fixed: float,
                 cost_verify_per_token: float = 0.0, k_min: int = 1, k_max: int = 16,
                 k_init: int = 4, decay: float = 0.9):
        if not 0.0 <= decay < 1.0:
            raise ValueError("decay must be in [0, 1)")
        self.costs = (cost_draft, cost_verify_fixed, cost_verify_per_token)
        self.k_min, self.k_max, self.decay = k_min, k_max, decay
        self.alpha = None
        self.k = int(min(max(k_init, k_min), k_max))

    def update(self, alpha) -> int:
        """Fold in one step's acceptance probabilities (a tensor, array or
        float; NaN entries ignored) and return the draft length to use next."""
        if isinstance(alpha, torch.Tensor):
            a = alpha.detach().float()
            a = a[~torch.isnan(a)]
            if a.numel() == 0:
                return self.k
            mean = float(a.mean())
        else:
            mean = float(alpha)
            if mean != mean:
                return self.k
        mean = min(max(mean, 0.0), 1.0)
        self.alpha = mean if self.alpha is None else self.decay * self.alpha + (1 - self.decay) * mean
        self.k = choose_k(self.alpha, *self.costs, k_min=self.k_min, k_max=self.k_max)
        return self.k


# specv_plan's kernel codes
KERNEL_NAMES = {0: "tile", 1: "rows-stream", 2: "rows-resident", 3: "tile-tma", 4: "rows-seq"}


def plan(B: int, K: int, V: int, dtype: int = F32, mode: int = PROB_MIX) -> dict:
    """The launch specv_verify would make (host-only query)."""
    kern, clus = ctypes.c_int32(0), ctypes.c_int32(0)
    ctas, ws = ctypes.c_int64(0), ctypes.c_int64(0)
    st = load().specv_plan(int(B), int(K), int(V), int(dtype), int(mode), ctypes.byref(kern),
                           ctypes.byref(clus), ctypes.byref(ctas), ctypes.byref(ws))
    _check(st, "specv_plan")
    flags = ctypes.c_uint32(0)
    _check(load().specv_plan_flags(int(B), int(K), int(V), int(dtype), int(mode),
                                   ctypes.byref(flags)), "specv_plan_flags")
    return dict(kernel=KERNEL_NAMES.get(kern.value, str(kern.value)), cluster=clus.value,
                ctas=ctas.value, workspace_bytes=ws.value,
                early_exit=bool(flags.value & 1), split_draws=bool(flags.value & 2))


def raw_call(name: str, *args) -> int:
    """Call an entry point of the C ABI with raw arguments (tests of the boundary)."""
    return int(getattr(load(), name)(*args))
