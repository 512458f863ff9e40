"""fp64 CPU oracle for the speculative-decoding verify/accept step (RAPID).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The CUDA library and its
Python binding never import it, and it imports nothing from them.

The arithmetic lives in ``specv_oracle.c`` (plain C, double precision, one
sequence at a time, following the per-step loop of the RAPID explainer's
"3) 候选验证机制（伪代码）" section).  This module compiles it with gcc, loads it
with ctypes and marshals numpy arrays.  ctypes releases the GIL during a
foreign call, so ``verify`` can split the batch over host threads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

PROB_MIX = 0
LOGIT_MIX = 1
GREEDY = 2

FLAG_INVALID = 1
FLAG_RESIDUAL_ZERO = 2
FLAG_CDF_FALLBACK = 4
FLAG_BONUS = 8

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (plain gcc)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        ip = ctypes.POINTER(ctypes.c_int32)
        i64 = ctypes.c_int64
        lib.oracle_softmax.argtypes = [dp, i64, dp]
        lib.oracle_softmax.restype = None
        lib.oracle_mix_prob.argtypes = [dp, dp, ctypes.c_double, i64, dp]
        lib.oracle_mix_prob.restype = None
        lib.oracle_mix_logit.argtypes = [dp, dp, ctypes.c_double, i64, dp]
        lib.oracle_mix_logit.restype = None
        lib.oracle_sample_inverse_cdf.argtypes = [dp, i64, ctypes.c_double,
                                                  ctypes.POINTER(ctypes.c_int), dp]
        lib.oracle_sample_inverse_cdf.restype = i64
        lib.oracle_rows.argtypes = [fp, fp, ctypes.c_int32, i64, ctypes.c_double,
                                    ctypes.c_int, dp, dp]
        lib.oracle_rows.restype = None
        lib.oracle_verify.argtypes = [fp, fp, ip, fp, fp, fp, i64, i64, ctypes.c_int32, i64,
                                      ctypes.c_int, ip, ip, dp, dp, dp, dp, dp, dp, ip]
        lib.oracle_verify.restype = ctypes.c_int
        lib.oracle_mix_logit_entry.argtypes = [ctypes.c_double] * 3
        lib.oracle_mix_logit_entry.restype = ctypes.c_double
        lib.oracle_greedy_scores.argtypes = [fp, fp, ctypes.c_float, i64, dp]
        lib.oracle_greedy_scores.restype = None
        lib.oracle_greedy_argmax.argtypes = [fp, fp, ctypes.c_float, i64, dp]
        lib.oracle_greedy_argmax.restype = i64
        lib.oracle_verify_greedy.argtypes = [fp, fp, ip, fp, i64, i64, ctypes.c_int32, i64, ip, ip,
                                             dp]
        lib.oracle_verify_greedy.restype = None
        lib.oracle_verify_tree.argtypes = [fp, fp, ip, ip, ip, fp, fp, fp, i64, i64,
                                           ctypes.c_int32, ctypes.c_int32, i64, ctypes.c_int, ip,
                                           ip, ip, dp, dp]
        lib.oracle_verify_tree.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _f32(a):
    """fp32 contiguous copy; torch bf16/fp32 tensors are widened exactly."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.int32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.int32)


def softmax(z) -> np.ndarray:
    z = _f64(z)
    out = np.empty_like(z)
    _load().oracle_softmax(_ptr(z, ctypes.c_double), z.size, _ptr(out, ctypes.c_double))
    return out


def mix_prob(pt, pq, lam: float) -> np.ndarray:
    pt, pq = _f64(pt), _f64(pq)
    out = np.empty_like(pt)
    _load().oracle_mix_prob(_ptr(pt, ctypes.c_double), _ptr(pq, ctypes.c_double), float(lam),
                            pt.size, _ptr(out, ctypes.c_double))
    return out


def mix_logit(zt, zq, lam: float) -> np.ndarray:
    zt, zq = _f64(zt), _f64(zq)
    out = np.empty_like(zt)
    _load().oracle_mix_logit(_ptr(zt, ctypes.c_double), _ptr(zq, ctypes.c_double), float(lam),
                             zt.size, _ptr(out, ctypes.c_double))
    return out


def sample_inverse_cdf(w, u: float):
    """Returns (index, fallback_used, margin); index -1 when sum(w) == 0."""
    w = _f64(w)
    fb = ctypes.c_int(0)
    margin = ctypes.c_double(0.0)
    idx = _load().oracle_sample_inverse_cdf(_ptr(w, ctypes.c_double), w.size, float(u),
                                            ctypes.byref(fb), ctypes.byref(margin))
    return int(idx), bool(fb.value), float(margin.value)


def rows(zt_seq, zq_seq, lam: float, mode: int = PROB_MIX):
    """p~ rows [K+1][V] (row K = target softmax) and q rows [K][V] of one sequence."""
    zt = _f32(zt_seq)
    zq = _f32(zq_seq)
    K1, V = zt.shape
    K = K1 - 1
    pt = np.empty((K + 1, V), np.float64)
    q = np.empty((max(K, 1), V), np.float64)
    _load().oracle_rows(_ptr(zt, ctypes.c_float), _ptr(zq, ctypes.c_float), K, V, float(lam),
                        int(mode), _ptr(pt, ctypes.c_double), _ptr(q, ctypes.c_double))
    return pt, q[:K]


class Result(dict):
    """Outputs and diagnostics of ``verify`` (attribute access for convenience)."""
    __getattr__ = dict.__getitem__


def verify(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lam,
           mode: int = PROB_MIX, diagnostics: bool = True, threads: int | None = None,
           seq_range: tuple[int, int] | None = None) -> Result:
    """Run the oracle on a batch.

    target_logits [B][K+1][V], draft_logits [B][K][V] (fp32 or bf16, numpy or
    torch; widened to fp32 exactly), draft_tokens int32 [B][K], u_accept fp32
    [B][K], u_resample fp32 [B], lam fp32 [B].  ``seq_range`` restricts the
    work to sequences [b0, b1) (other rows of the outputs stay untouched).
    """
    zt = _f32(target_logits)
    zq = _f32(draft_logits)
    tok = _i32(draft_tokens)
    ua = _f32(u_accept)
    ur = _f32(u_resample).reshape(-1)
    lm = _f32(lam).reshape(-1)
    B, K1, V = zt.shape
    K = K1 - 1
    if zq.size == 0:
        zq = np.zeros((B, max(K, 0), V), np.float32)
    assert zq.shape == (B, K, V) and tok.shape == (B, K) and ua.shape == (B, K)
    assert ur.shape == (B,) and lm.shape == (B,)
    b0, b1 = seq_range if seq_range is not None else (0, B)
    out_tok = np.full((B, K + 1), -2, np.int32)
    out_n = np.full((B,), -2, np.int32)
    diag = {}
    if diagnostics:
        for name in ("ratio", "ptilde_x", "q_x", "alpha"):
            diag[name] = np.full((B, K), np.nan, np.float64)
        diag["accept_margin"] = np.full((B,), np.nan, np.float64)
        diag["cdf_margin"] = np.full((B,), np.nan, np.float64)
        diag["flags"] = np.zeros((B,), np.int32)
    lib = _load()
    dp = ctypes.c_double
    args_tail = (
        _ptr(diag.get("ratio"), dp), _ptr(diag.get("ptilde_x"), dp), _ptr(diag.get("q_x"), dp),
        _ptr(diag.get("alpha"), dp), _ptr(diag.get("accept_margin"), dp),
        _ptr(diag.get("cdf_margin"), dp), _ptr(diag.get("flags"), ctypes.c_int32))

    def run(lo, hi):
        rc = lib.oracle_verify(_ptr(zt, ctypes.c_float), _ptr(zq, ctypes.c_float),
                               _ptr(tok, ctypes.c_int32), _ptr(ua, ctypes.c_float),
                               _ptr(ur, ctypes.c_float), _ptr(lm, ctypes.c_float), lo, hi, K, V,
                               int(mode), _ptr(out_tok, ctypes.c_int32),
                               _ptr(out_n, ctypes.c_int32), *args_tail)
        if rc != 0:
            raise MemoryError("oracle_verify could not allocate its row buffers")

    nthreads = threads if threads is not None else (os.cpu_count() or 1)
    nthreads = max(1, min(nthreads, b1 - b0))
    if nthreads == 1:
        run(b0, b1)
    else:
        edges = np.linspace(b0, b1, nthreads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(lambda j: run(int(edges[j]), int(edges[j + 1])), range(nthreads)))
    res = Result(tokens=out_tok, n_accepted=out_n, threads=nthreads)
    res.update(diag)
    return res


def mix_logit_entry(zt: float, zq: float, lam: float) -> float:
    """One entry of (1 - lam) z_t + lam z_q with the masking rule (a -inf
    logit of positive weight gives -inf; a term of weight zero drops out)."""
    return float(_load().oracle_mix_logit_entry(float(zt), float(zq), float(lam)))


def greedy_scores(zt_row, zq_row, lam: float) -> np.ndarray:
    """The fp64 greedy scores w = (1 - lam) z_t + lam z_q of one row (zq_row
    None: w = z_t), with lam taken as the fp32 value the kernels read."""
    zt = _f32(zt_row).reshape(-1)
    zq = None if zq_row is None else _f32(zq_row).reshape(-1)
    out = np.empty(zt.size, np.float64)
    _load().oracle_greedy_scores(_ptr(zt, ctypes.c_float), _ptr(zq, ctypes.c_float),
                                 float(np.float32(lam)), zt.size, _ptr(out, ctypes.c_double))
    return out


def greedy_argmax(zt_row, zq_row, lam: float, with_gap: bool = False):
    """Argmax of the fp64 greedy scores of one row (zq_row None: w = z_t), the
    first index among equal maxima; with_gap also returns the relative gap
    (w_best - w_second) / max |logit| of the row."""
    zt = _f32(zt_row).reshape(-1)
    zq = None if zq_row is None else _f32(zq_row).reshape(-1)
    gap = ctypes.c_double(0.0)
    idx = int(_load().oracle_greedy_argmax(_ptr(zt, ctypes.c_float), _ptr(zq, ctypes.c_float),
                                           float(np.float32(lam)), zt.size, ctypes.byref(gap)))
    return (idx, float(gap.value)) if with_gap else idx


def verify_greedy(target_logits, draft_logits, draft_tokens, lam,
                  threads: int | None = None) -> Result:
    """Greedy verification of a batch (same layouts as ``verify``).  Returns
    tokens, n_accepted and tie_margin [B]: the smallest relative gap between
    the best and second-best fp64 score over the mixed rows the decision read
    (+inf if none)."""
    zt = _f32(target_logits)
    zq = _f32(draft_logits)
    tok = _i32(draft_tokens)
    lm = _f32(lam).reshape(-1)
    B, K1, V = zt.shape
    K = K1 - 1
    assert zq.shape == (B, K, V) and tok.shape == (B, K) and lm.shape == (B,)
    out_tok = np.full((B, K + 1), -2, np.int32)
    out_n = np.full((B,), -2, np.int32)
    margin = np.full((B,), np.nan, np.float64)
    lib = _load()

    def run(lo, hi):
        lib.oracle_verify_greedy(_ptr(zt, ctypes.c_float), _ptr(zq, ctypes.c_float),
                                 _ptr(tok, ctypes.c_int32), _ptr(lm, ctypes.c_float), lo, hi, K,
                                 V, _ptr(out_tok, ctypes.c_int32), _ptr(out_n, ctypes.c_int32),
                                 _ptr(margin, ctypes.c_double))

    nthreads = threads if threads is not None else (os.cpu_count() or 1)
    nthreads = max(1, min(nthreads, B))
    if nthreads == 1:
        run(0, B)
    else:
        edges = np.linspace(0, B, nthreads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(lambda j: run(int(edges[j]), int(edges[j + 1])), range(nthreads)))
    return Result(tokens=out_tok, n_accepted=out_n, tie_margin=margin, threads=nthreads)


def verify_tree(target_logits, draft_logits, parent, draft_row, tokens, u_accept, u_resample,
                lam, mode: int = PROB_MIX, threads: int | None = None) -> Result:
    """Tree verification (the reading in specv_oracle.c).  target_logits
    [B][N+1][V], draft_logits [B][M][V], parent/draft_row/tokens int32 [B][N+1],
    u_accept fp32 [B][N+1], u_resample and lam fp32 [B].  Returns tokens and
    path [B][N+1], n_accepted [B], accept_margin and cdf_margin [B]."""
    zt = _f32(target_logits)
    zq = _f32(draft_logits)
    par, drow, tok = _i32(parent), _i32(draft_row), _i32(tokens)
    ua = _f32(u_accept)
    ur = _f32(u_resample).reshape(-1)
    lm = _f32(lam).reshape(-1)
    B, N1, V = zt.shape
    N = N1 - 1
    if zq.ndim != 3 or zq.shape[0] != B or (zq.shape[1] > 0 and zq.shape[2] != V):
        raise ValueError("draft_logits must be [B][M][V]")
    M = zq.shape[1]
    if M == 0:
        zq = np.zeros((B, 1, V), np.float32)
    for a in (par, drow, tok, ua):
        assert a.shape == (B, N + 1)
    out_tok = np.full((B, N + 1), -2, np.int32)
    out_path = np.full((B, N + 1), -2, np.int32)
    out_n = np.full((B,), -2, np.int32)
    am = np.full((B,), np.nan, np.float64)
    cm = np.full((B,), np.nan, np.float64)
    lib = _load()
    dp_ = ctypes.c_double

    def run(lo, hi):
        rc = lib.oracle_verify_tree(
            _ptr(zt, ctypes.c_float), _ptr(zq, ctypes.c_float), _ptr(par, ctypes.c_int32),
            _ptr(drow, ctypes.c_int32), _ptr(tok, ctypes.c_int32), _ptr(ua, ctypes.c_float),
            _ptr(ur, ctypes.c_float), _ptr(lm, ctypes.c_float), lo, hi, N, M, V, int(mode),
            _ptr(out_tok, ctypes.c_int32), _ptr(out_path, ctypes.c_int32),
            _ptr(out_n, ctypes.c_int32), _ptr(am, dp_), _ptr(cm, dp_))
        if rc != 0:
            raise MemoryError("oracle_verify_tree could not allocate its row buffers")

    nthreads = threads if threads is not None else (os.cpu_count() or 1)
    nthreads = max(1, min(nthreads, B))
    if nthreads == 1:
        run(0, B)
    else:
        edges = np.linspace(0, B, nthreads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(lambda j: run(int(edges[j]), int(edges[j + 1])), range(nthreads)))
    return Result(tokens=out_tok, path=out_path, n_accepted=out_n, accept_margin=am,
                  cdf_margin=cm, threads=nthreads)
