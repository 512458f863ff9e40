"""Benchmark of the verify/accept step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 4] [--mode prob|logit]
    python bench.py --impl reference ...      # the fp64 CPU oracle, timed on the host cores

A step is one specv_verify call over the whole batch of the chosen workload
(default: B=256 sequences, K=8 drafts, V=128256, fp32 logits -- the batched
128K-vocabulary workload).  The metric is verified draft rows per second,
B*K per step; the roofline line reports the achieved HBM bandwidth of the
verify kernel with the algorithmic bytes (2K+1)*B*V*sizeof(dtype) per launch.
The inputs (2.2 GB) are larger than L2, so no flush is needed between steps.

Under torchrun (N > 1) one global batch of N x B sequences is split by rank
into contiguous shards of B sequences (the library's specv_shard_bounds), each
verified on its rank's GPU with no collective in the data path (weak scaling:
the per-GPU batch is fixed); after the timed region the shards' outputs are
gathered in order into the global batch's.  The reported value is all ranks'
rows over the slowest rank's time.

The line also carries `per_config`: the other workloads (B=1 Llama-shaped,
B=32 Qwen-shaped, the 10^6-sequence exactness workload) and the batched
workload reading every row, each timed the same way.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "verified draft rows/sec (B·K) and achieved HBM GB/s vs GB300 peak, 1 GPU"
UNIT = "rows/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = [os.path.join(ROOT, "speculative_decoding_verification_specv_gb300", "csrc", f)
                  for f in ("specv_rows.cu", "specv_device.cuh", "specv_block.cuh",
                            "specv_segments.cuh", "specv_stream.cuh", "specv_internal.h")]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="specv", choices=["specv", "reference"])
    ap.add_argument("--config", type=int, default=4, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--mode", default="prob", choices=["prob", "logit", "greedy"],
                    help="sampling rule with the probability or logit mixture, or greedy")
    ap.add_argument("--B", type=int, default=None, help="override the batch size (profiling)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every step from the host instead of replaying a CUDA graph")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-api", default="direct", choices=["direct", "early-exit", "chunked"],
                    help="host-buffer call of the e2e leg: specv_verify_host_direct (kernels read "
                         "the pinned inputs in place), specv_verify_host_early_exit (copies the "
                         "rows the step reaches) or specv_verify_host (copies every row)")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="chunks of the host-buffer call (0 = the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config block (the other workloads, timed the same way)")
    ap.add_argument("--tree", default=None, metavar="SHAPE",
                    help="time specv_verify_tree on a draft tree of this shape (chain, kary:k, "
                         "star, random:f) with --tree-nodes nodes besides the root")
    ap.add_argument("--tree-nodes", type=int, default=14)
    ap.add_argument("--stats", action="store_true",
                    help="time specv_acceptance_rates (exact acceptance probabilities of every "
                         "drafted position) instead of the verify step")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws, device):
    """The largest value of x over all ranks (the slowest rank's time); x on one
    rank is returned unchanged."""
    if ws == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def global_batch_slice(w, n_shards, lo, hi, device):
    """Sequences [lo, hi) of the global batch of n_shards * w.B sequences: the
    concatenation of n_shards seeded batches of workload w (sub-batch j drawn
    with seed offset j), so that any contiguous shard is reproducible on its
    own rank."""
    B = w.B
    parts = []
    for j in range(lo // B, max(lo // B + 1, (hi + B - 1) // B)):
        x = workloads.make_inputs(w, device, seed_offset=j)
        a, b = max(lo - j * B, 0), max(min(hi - j * B, B), 0)
        parts.append({k: v[a:b] for k, v in x.items()})
    return {k: torch.cat([p[k] for p in parts]).contiguous() for k in parts[0]}


def gather_shards(tokens, n_accepted, ws):
    """Every rank's output rows, concatenated in rank order (the shards are
    contiguous and in order, so this is the global batch's output)."""
    import numpy as np
    t = tokens.cpu().numpy() if hasattr(tokens, "cpu") else np.asarray(tokens)
    n = n_accepted.cpu().numpy() if hasattr(n_accepted, "cpu") else np.asarray(n_accepted)
    if ws == 1:
        return t, n
    import torch.distributed as dist
    objs = [None] * ws
    dist.all_gather_object(objs, (t, n))
    return np.concatenate([o[0] for o in objs]), np.concatenate([o[1] for o in objs])


def job_throughput(rows_per_step, steps, ws, slowest_ms):
    """Whole-job rows/s: every rank verifies rows_per_step rows per step (weak
    scaling), all ranks' rows over the slowest rank's time."""
    return rows_per_step * steps * ws / (slowest_ms / 1e3)


# kernel function timed for the roofline, by the planner's kernel name
PLAN_KERNEL_FUNCTION = {"tile": "tile_kernel", "rows-stream": "rows_kernel",
                        "rows-resident": "resident_kernel", "tile-tma": "tile_tma_kernel",
                        "rows-seq": "rows_seq_kernel"}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def needed_bytes(n_accepted, K, V, elem):
    """Bytes of logits the verify step needs when it stops at the first
    rejection: the row pairs of positions 0..n and, when every draft passes,
    the bonus row -- (2 min(n + 1, K) + [n = K]) V s per sequence.  An invalid
    sequence (n < 0) is counted with every row."""
    n = torch.as_tensor(n_accepted).to(torch.int64).cpu()
    rows = torch.where(n < 0, torch.full_like(n, 2 * K + 1),
                       2 * torch.clamp(n + 1, max=K) + (n == K).to(torch.int64))
    return int(rows.sum().item()) * V * elem


def capture_graph(launch, dev):
    """A CUDA graph of one launch() call, captured on a side stream after one
    plain call on that same stream: the library keeps its scratch per stream
    and creates it on the first call, so the captured graph holds the verify
    launches only (no allocation or clearing nodes), as it would for a user
    who calls once before capturing."""
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        launch()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch()
    torch.cuda.synchronize(dev)
    return graph


def kernel_source_hash():
    """Hash of the row kernels' code: comments and whitespace are left out, so
    that a profile's traffic stays attached to the code it was measured on."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)  # block comments
        text = re.sub(r"//[^\n]*", " ", text)                # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(config_name, mode="prob"):
    """DRAM bytes per launch from a committed ncu summary under profiles/ taken
    on the current kernel source for this workload and mode; else None."""
    import glob
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        try:
            text = open(path).read()
        except OSError:
            continue
        vals = {}
        for line in text.splitlines():
            if line.startswith("bench-key ") and ":" in line:
                k, v = line[len("bench-key "):].split(":", 1)
                vals[k.strip()] = v.strip()
        if (vals.get("kernel_source_sha256_16") != kernel_source_hash()
                or vals.get("workload") != config_name or vals.get("mode", "prob") != mode):
            continue
        try:
            return int(vals["dram_bytes_per_launch"])
        except (KeyError, ValueError):
            continue
    return None


class L2Flush:
    """Evicts the previous step's inputs from L2 between timed steps (outside
    the step's events): a 2x-L2 buffer is written, then a second 2x-L2 buffer
    is read, so that the written lines are written back to HBM here and the
    timed step starts with a clean L2 that holds none of its inputs."""

    def __init__(self, dev, l2_bytes):
        n = 2 * l2_bytes // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.zeros(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, i):
        self.w.fill_(float(i))
        torch.sum(self.r, dim=0, out=self.sink)


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


MODES = {"prob": 0, "logit": 1, "greedy": 2}


def oracle_step(xh, mode, threads):
    """One oracle pass over a host batch (the sampling rule, or greedy)."""
    import oracle
    if mode == MODES["greedy"]:
        oracle.verify_greedy(xh["target_logits"], xh["draft_logits"], xh["draft_tokens"],
                             xh["lam"], threads=threads)
    else:
        oracle.verify(xh["target_logits"], xh["draft_logits"], xh["draft_tokens"],
                      xh["u_accept"], xh["u_resample"], xh["lam"], mode=mode,
                      diagnostics=False, threads=threads)


def cpu_baseline(w, mode, target_seconds, host_inputs=None):
    """The fp64 oracle, as it stands, on a bounded sample of the workload."""
    import oracle
    oracle.build()
    if host_inputs is None:
        nb = min(w.B, 16)
        host_inputs = workloads.make_inputs(w.scaled(B=nb), "cpu")
    xh = host_inputs
    B = xh["target_logits"].shape[0]
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    passes = 0
    seqs = 0
    while True:
        oracle_step(xh, mode, threads)
        passes += 1
        seqs += B
        el = time.perf_counter() - t0
        if el >= target_seconds or passes >= 5000:
            break
    rows = seqs * w.K
    return {"value": rows / el, "unit": UNIT, "cores": min(threads, B), "kind": "oracle",
            "sample": f"{passes} pass(es) over {B} sequences of {w.name} (K={w.K}, V={w.V}, "
                      f"{w.dtype}); {el:.1f} s wall on {min(threads, B)} host threads"}


def launches_per_step(plan):
    """Kernel launches of one specv_verify call under this plan."""
    return 2 if plan.get("split_draws") else 1


def time_verify(specv, w, mode, dev, steps, warmup, l2_bytes):
    """Mean device time (ms) of one specv_verify call on workload w: a CUDA
    graph of the call replayed between CUDA events on its stream, the L2
    flushed before every step when the inputs are smaller than twice the L2.
    Returns (ms, mean n_accepted, outputs)."""
    x = workloads.make_inputs(w, dev)
    out_tok = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((w.B,), dtype=torch.int32, device=dev)
    args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
            x["u_resample"], x["lam"])
    graph = capture_graph(lambda: specv.verify(*args, mode=mode, out_tokens=out_tok,
                                               out_n_accepted=out_n,
                                               stream=torch.cuda.current_stream(dev)), dev)
    flush = L2Flush(dev, l2_bytes) if w.roofline_bytes < 2 * l2_bytes else None
    stream = torch.cuda.current_stream(dev)
    for i in range(max(3, warmup)):
        if flush is not None:
            flush(i)
        graph.replay()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush(i)
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return ms, float(out_n.float().mean().item()), (out_tok, out_n), flush is not None


# the per_config block: (workload, mode, environment, steps)
PER_CONFIG = [(2, "prob", {}, 400), (3, "prob", {}, 400), (5, "prob", {}, 200),
              (4, "prob", {"SPECV_EARLY_EXIT": "0"}, 100)]


def run_per_config(specv, dev, args, l2_bytes):
    """The other workloads (and the batched one reading every row), each timed
    like the headline step, with its rows/s and HBM fraction."""
    peak, _ = measured_peak()
    out = []
    for cfg, mname, env, steps in PER_CONFIG:
        w = workloads.WORKLOADS[cfg]
        mode = MODES[mname]
        old = {k: os.environ.get(k) for k in env}
        os.environ.update(env)
        try:
            plan = specv.plan(w.B, w.K, w.V, 1 if w.dtype == "bf16" else 0, mode)
            ms, mean_n, (_, n), flushed = time_verify(specv, w, mode, dev, steps, args.warmup,
                                                      l2_bytes)
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        alg = (needed_bytes(n, w.K, w.V, w.elem_bytes) if plan.get("early_exit")
               else w.roofline_bytes)
        gbs = alg / (ms / 1e3) / 1e9
        out.append({"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "logits": w.dtype,
                    "mode": mname, "env": env, "us_per_step": ms * 1e3,
                    "rows_per_s": w.B * w.K / (ms / 1e3), "algorithmic_bytes": alg,
                    "hbm_gbs": gbs, "frac": gbs / peak, "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
                    "every_row_frac": w.roofline_bytes / (ms / 1e3) / 1e9 / peak,
                    "traffic": profiled_traffic(w.name, mname) if not env else None,
                    "mean_accepted": mean_n, "plan": plan, "steps": steps,
                    "gpu_launches": steps * launches_per_step(plan),
                    "l2": "flushed before every step" if flushed else "inputs > L2"})
        torch.cuda.empty_cache()
    return out


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.config]
    mode = MODES[args.mode]
    import oracle
    oracle.build()
    nb = min(w.B, 8)
    xh = workloads.make_inputs(w.scaled(B=nb), "cpu")
    threads = os.cpu_count() or 1

    def step():
        oracle_step(xh, mode, threads)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    rows = nb * w.K * args.steps
    value = rows / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "logits": w.dtype,
                   "mode": args.mode, "sample_sequences_per_step": nb},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(threads, nb), "kind": "oracle",
                         "sample": f"{nb} sequences of {w.name} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_stats(args):
    """One line for the acceptance-probability kernel: drafted positions per
    second, and its HBM bandwidth with the algorithmic bytes 2K*B*V*s (every
    drafted row pair read once; the second pass is meant to hit L2)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import speculative_decoding_verification_specv_gb300 as specv
    specv.load(build_if_missing=True)
    w = workloads.WORKLOADS[args.config]
    if args.B:
        w = w.scaled(B=args.B, name=f"{w.name}-B{args.B}")
    mode = MODES[args.mode]
    x = workloads.make_inputs(w, dev)
    out = torch.empty((w.B, w.K), dtype=torch.float32, device=dev)

    def launch():
        specv.acceptance_rates(x["target_logits"], x["draft_logits"], x["lam"], mode=mode,
                               out=out, stream=torch.cuda.current_stream(dev))
    graph = capture_graph(launch, dev)
    stream = torch.cuda.current_stream(dev)
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    elem = 2 if w.dtype == "bf16" else 4
    alg = 2 * w.K * w.B * w.V * elem
    flush = L2Flush(dev, l2) if alg < 2 * l2 else None
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        for i in range(args.steps):
            if flush is not None:
                flush(i)
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    peak, kind = measured_peak()
    achieved = alg / (ms / 1e3) / 1e9
    line = {
        "metric": "drafted positions/s with exact acceptance probability (specv_acceptance_rates)",
        "value": w.B * w.K / (ms / 1e3), "unit": "positions/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "dtype": "f32" if w.dtype == "f32" else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "mode": args.mode,
                   "l2": "flushed before every step" if flush is not None else "inputs > L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": alg, "kernel": "alpha_kernel",
                     "peak_source": kind},
        "clocks": clk.summary(), "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def run_tree(args):
    """One line for tree verification: tree nodes verified per second, and the
    HBM bandwidth of the call with the bytes of one read of every node's rows
    (target rows of all nodes, draft rows of the nodes with children); the walk
    reads the rows of the nodes it visits again, which this figure leaves out."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import speculative_decoding_verification_specv_gb300 as specv
    specv.load(build_if_missing=True)
    w = workloads.WORKLOADS[args.config]
    B = args.B or w.B
    N = args.tree_nodes
    mode = MODES[args.mode]
    if mode == MODES["greedy"]:
        raise SystemExit("tree verification takes prob or logit mode")
    x = workloads.make_tree_inputs(B, N, w.V, w.dtype, args.tree, lam=float(w.lam[0])
                                   if w.lam[0] != "uniform" else 0.25, device=dev)
    M = x["draft_logits"].shape[1]
    elem = 2 if w.dtype == "bf16" else 4
    alg = (N + 1 + M) * B * w.V * elem
    args_t = (x["target_logits"], x["draft_logits"], x["parent"], x["draft_row"], x["tokens"],
              x["u_accept"], x["u_resample"], x["lam"])
    res = {}

    def launch():
        res["out"] = specv.verify_tree(*args_t, mode=mode)
    graph = capture_graph(launch, dev)
    out = res["out"]
    stream = torch.cuda.current_stream(dev)
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    flush = L2Flush(dev, l2) if alg < 2 * l2 else None
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        for i in range(args.steps):
            if flush is not None:
                flush(i)
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    peak, kind = measured_peak()
    achieved = alg / (ms / 1e3) / 1e9
    line = {
        "metric": "draft-tree nodes verified/s (specv_verify_tree)",
        "value": B * N / (ms / 1e3), "unit": "nodes/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "dtype": "f32" if w.dtype == "f32" else "bf16", "data": "synthetic",
        "config": {"workload": f"tree-{args.tree}-n{N}-v{w.V}-{w.dtype}-b{B}", "B": B, "N": N,
                   "M": M, "V": w.V, "mode": args.mode,
                   "mean_accepted": float(out[2].float().mean().item()),
                   "l2": "flushed before every step" if flush is not None else "inputs > L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": alg, "kernel": "tree_kernel",
                     "peak_source": kind},
        "clocks": clk.summary(), "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.tree:
        run_tree(args)
        return
    if args.stats:
        run_stats(args)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import speculative_decoding_verification_specv_gb300 as specv
    specv.load(build_if_missing=True)

    w = workloads.WORKLOADS[args.config]
    if args.B:
        w = w.scaled(B=args.B, name=f"{w.name}-B{args.B}")
    mode = MODES[args.mode]
    # this rank's shard of one global batch of ws x B sequences
    B_global = ws * w.B
    shard_lo, shard_hi = specv.shard_bounds(B_global, ws, rank)
    x = global_batch_slice(w, ws, shard_lo, shard_hi, dev)
    stream = torch.cuda.current_stream(dev)
    out_tok = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((w.B,), dtype=torch.int32, device=dev)
    call_args = (x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
                 x["u_resample"], x["lam"])

    def launch():
        specv.verify(*call_args, mode=mode, out_tokens=out_tok, out_n_accepted=out_n,
                     stream=torch.cuda.current_stream(dev))

    # One step = one specv_verify call.  By default it is captured once in a
    # CUDA graph (the verify launches only: the stream's scratch exists before
    # the capture) and replayed, so the device time is not hidden behind host
    # launch overhead.
    graph = None
    if not args.no_graph:
        graph = capture_graph(launch, dev)

    def step():
        if graph is not None:
            graph.replay()
        else:
            launch()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    # Working sets smaller than twice the L2 are re-read from L2 by the next
    # step; for those the L2 is flushed (a 2x-L2 buffer is written) before
    # every timed step, outside the per-step events.
    try:
        l2_bytes = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        l2_bytes = 126 * 2**20
    flush_buf = None
    if w.roofline_bytes < 2 * l2_bytes:
        flush_buf = L2Flush(dev, l2_bytes)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for i in range(K):
            if flush_buf is not None:
                flush_buf(i)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    clk_summary = clk.summary()
    total_ms = t_start.elapsed_time(t_end)
    per_call_ms = [a.elapsed_time(b) for a, b in ev]
    if flush_buf is not None:  # the timed region holds the flushes: count the steps only
        total_ms = sum(per_call_ms)
    total_ms = max_over_ranks(total_ms, ws, dev)
    rows_per_step = w.B * w.K
    value = job_throughput(rows_per_step, K, ws, total_ms)
    # the shards' outputs, concatenated in order: the global batch's outputs
    _, n_global = gather_shards(out_tok, out_n, ws)
    mean_accepted = float(n_global.astype("float64").mean())

    # end to end: pinned host inputs -> device, verify, result -> host, every step
    e2e = None
    if not args.no_e2e:
        host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in x.items()}
        for k, v in x.items():
            host[k].copy_(v)
        host_tok = torch.empty((w.B, w.K + 1), dtype=torch.int32, pin_memory=True)
        host_n = torch.empty((w.B,), dtype=torch.int32, pin_memory=True)
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = host_tok.numel() * 4 + host_n.numel() * 4
        del x  # the device copies of the inputs: the host call stages its own

        link = {}

        def e2e_step():
            # one C-ABI call on host buffers, then the results back to the host
            if args.e2e_api == "direct":
                # the kernels read the page-locked inputs over the host link in place
                specv.verify_host_direct(
                    host["target_logits"], host["draft_logits"], host["draft_tokens"],
                    host["u_accept"], host["u_resample"], host["lam"], mode=mode,
                    out_tokens=host_tok, out_n_accepted=host_n, stream=stream)
            elif args.e2e_api == "early-exit":
                # position by position, only the rows the verify step reaches
                _, _, link["h2d"], link["d2h"] = specv.verify_host_early_exit(
                    host["target_logits"], host["draft_logits"], host["draft_tokens"],
                    host["u_accept"], host["u_resample"], host["lam"], mode=mode,
                    out_tokens=host_tok, out_n_accepted=host_n, stream=stream)
            else:
                # every row, in chunks whose copies overlap the verify launches
                specv.verify_host(host["target_logits"], host["draft_logits"],
                                  host["draft_tokens"], host["u_accept"], host["u_resample"],
                                  host["lam"], mode=mode, out_tokens=host_tok,
                                  out_n_accepted=host_n, chunks=args.e2e_chunks, stream=stream)
                link["h2d"], link["d2h"] = h2d, d2h
        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        e_steps = max(3, min(K, 10))
        barrier()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e_ms = max_over_ranks(a.elapsed_time(b), ws, dev)
        if args.e2e_api == "direct":
            # what crosses the host link: the per-sequence arrays and the rows
            # the outputs depend on (the token draws read their rows a second
            # time from a device copy the stream fills); left out: the part of
            # a position streamed before an earlier rejection of its sequence
            # was published.  The outputs are written in place.
            n_h = host_n.to(torch.int64)
            link["h2d"] = (needed_bytes(n_h, w.K, w.V, w.elem_bytes) +
                           sum(host[k].numel() * host[k].element_size()
                               for k in ("draft_tokens", "u_accept", "u_resample", "lam")))
            link["d2h"] = d2h
        e2e = {"value": job_throughput(rows_per_step, e_steps, ws, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": link["h2d"], "d2h_bytes_per_step": link["d2h"],
               "every_row_h2d_bytes": h2d, "steps": e_steps, "ms_per_step": e_ms / e_steps,
               "api": {"direct": "specv_verify_host_direct (pinned host buffers read and "
                                 "written in place by the kernels over the host link; only "
                                 "the rows the step reaches cross it)",
                       "early-exit": "specv_verify_host_early_exit (pinned host buffers; rows "
                                     "copied position by position up to each sequence's "
                                     "first rejection)",
                       "chunked": "specv_verify_host (pinned host buffers, chunks="
                                  f"{args.e2e_chunks or 'auto'})"}[args.e2e_api]}
        del host

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    plan = specv.plan(w.B, w.K, w.V, 1 if w.dtype == "bf16" else 0, mode)
    kern_ms = statistics.mean(per_call_ms)
    # With early exit the step reads only the rows the outputs depend on, so
    # the algorithmic bytes are those rows (from the outputs of this run);
    # every row read once, (2K+1)BVs, is reported beside them.
    all_rows = w.roofline_bytes
    alg_bytes = needed_bytes(out_n, w.K, w.V, w.elem_bytes) if plan.get("early_exit") else all_rows
    achieved = alg_bytes / (kern_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    traffic = profiled_traffic(w.name, args.mode)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                "kernel": ("rows_greedy_kernel" if args.mode == "greedy" and
                           plan["kernel"] == "rows-stream" else
                           PLAN_KERNEL_FUNCTION.get(plan["kernel"], plan["kernel"])),
                "algorithmic_bytes_per_launch": alg_bytes,
                "algorithmic_bytes": ("rows up to the first rejection (early exit): "
                                      "(2 min(n+1, K) + [n = K]) V s per sequence"
                                      if plan.get("early_exit") else
                                      "every logit read once: (2K+1) B V s"),
                "all_rows_bytes_per_launch": all_rows,
                "frac_at_all_rows_bytes": all_rows / (kern_ms / 1e3) / 1e9 / peak,
                "launch_ms_mean": kern_ms, "launch_ms_min": min(per_call_ms),
                "timing": ("CUDA events around each replay of a CUDA graph holding one "
                           "specv_verify call" if graph is not None else
                           "CUDA events around each specv_verify call") +
                          " on its stream (the verify launches only)",
                # the roofline as the task states it: every logit read once,
                # (2K+1) B V s per launch, whatever the kernel skips
                "every_row_read_once": {
                    "bytes_per_launch": all_rows,
                    "gbs": all_rows / (kern_ms / 1e3) / 1e9,
                    "frac_of_measured": all_rows / (kern_ms / 1e3) / 1e9 / peak,
                    "frac_of_nominal_8tbs": all_rows / (kern_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                    "note": ("with early exit the kernel reads only the rows the outputs depend "
                             "on, so this rate can exceed the copy peak; `frac` above is the "
                             "bandwidth over those rows" if plan.get("early_exit") else
                             "equal to `frac`: every row is read")}}
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline(w, mode, args.cpu_seconds)
    per_config = None
    if not args.no_per_config and ws == 1 and args.B is None:
        with ClockSampler(local) as pclk:
            per_config = {"workloads": run_per_config(specv, dev, args, l2_bytes)}
        per_config["clocks"] = pclk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if w.dtype == "f32" else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "logits": w.dtype,
                   "mode": args.mode, "lambda": list(w.lam), "structure": w.structure,
                   "plan": plan, "graph_replay": graph is not None,
                   "l2": "L2 flushed before every timed step (2x-L2 write, then a 2x-L2 "
                         "read, outside the step events)" if flush_buf is not None else
                         "inputs larger than L2 (no flush)",
                   "global_batch": B_global,
                   "parallelism": (f"one global batch of {B_global} sequences split into {ws} "
                                   f"contiguous shards of {w.B}, one per GPU" if ws > 1 else
                                   "1 GPU")},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk_summary,
        "gpu_launches": K * launches_per_step(plan), "mean_accepted": mean_accepted,
        "hbm_gbs_step": alg_bytes * ws / (total_ms / K / 1e3) / 1e9,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
