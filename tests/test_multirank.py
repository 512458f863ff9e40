"""The N>1 host path of the benchmark: replicas with weak scaling.

Every rank verifies its own batch on its own GPU; nothing in the data path is
exchanged.  Across ranks only the timing is combined: the job's time is the
slowest rank's, and the job's throughput counts every rank's rows over that
time.  These tests run the combination as two gloo ranks on the CPU, and check
that the reference arm does its work on rank 0 alone.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, times, out_path):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        slowest = bench.max_over_ranks(times[rank], ws, "cpu")
        value = bench.job_throughput(100, 10, ws, slowest)
        dist.barrier()
        if rank == 0:
            with open(out_path, "w") as f:
                f.write(f"{slowest!r} {value!r}\n")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(3.0, 5.0), (7.5, 2.0)])
def test_two_gloo_ranks_take_the_slowest_time(tmp_path, times):
    ws = 2
    out = tmp_path / "result.txt"
    mp.start_processes(_rank_main, args=(ws, _free_port(), list(times), str(out)), nprocs=ws,
                       join=True, start_method="spawn")
    slowest, value = (float(v) for v in out.read_text().split())
    assert slowest == max(times)
    # 100 rows per step on each rank, 10 steps, 2 ranks, over the slowest rank's ms
    assert value == pytest.approx(100 * 10 * 2 / (max(times) / 1e3), rel=1e-12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.25, 1, "cpu") == 4.25
    assert bench.job_throughput(2048, 3, 1, 1.5) == pytest.approx(2048 * 3 / 1.5e-3)


def test_ranks_draw_distinct_inputs():
    """Each rank verifies its own seeded batch (seed offset = rank)."""
    w = workloads.WORKLOADS[1]
    a = workloads.make_inputs(w, "cpu", seed_offset=0)
    b = workloads.make_inputs(w, "cpu", seed_offset=1)
    a2 = workloads.make_inputs(w, "cpu", seed_offset=0)
    assert not torch.equal(a["target_logits"], b["target_logits"])
    for k in a:
        assert torch.equal(a[k], a2[k])


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--config", "1"],
                       env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_plan_kernel_names_map_to_kernel_functions():
    import speculative_decoding_verification_specv_gb300 as specv
    names = getattr(specv, "KERNEL_NAMES", None)
    if names is None:
        pytest.skip("binding exposes no kernel-name table")
    for name in names.values():
        assert name in bench.PLAN_KERNEL_FUNCTION


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_oracle_step_runs_every_mode(mode):
    """The oracle leg of the benchmark (cpu_baseline and the reference arm)."""
    w = workloads.WORKLOADS[1]
    xh = workloads.make_inputs(w, "cpu")
    bench.oracle_step(xh, mode, 2)
    out = bench.cpu_baseline(w, mode, 0.05, host_inputs=xh)
    assert out["kind"] == "oracle" and out["value"] > 0


def test_l2_flush_runs_on_any_device():
    """The between-steps L2 flush (write a 2x-L2 buffer, then read another)."""
    f = bench.L2Flush("cpu", 1 << 16)
    f(3)
    assert float(f.w[0]) == 3.0 and float(f.sink) == 0.0


def test_needed_bytes_of_early_exit():
    """The benchmark's algorithmic bytes under early exit: the row pairs of
    positions 0..n and, when every draft passes, the bonus row; an invalid
    sequence counts every row."""
    K, V, s = 8, 10, 4
    n = torch.tensor([0, 3, 8, -1], dtype=torch.int32)
    rows = 2 * 1 + 2 * 4 + (2 * 8 + 1) + (2 * 8 + 1)
    assert bench.needed_bytes(n, K, V, s) == rows * V * s
    # every sequence accepting all drafts needs every row: (2K+1) B V s
    allk = torch.full((5,), K, dtype=torch.int32)
    assert bench.needed_bytes(allk, K, V, s) == (2 * K + 1) * 5 * V * s
