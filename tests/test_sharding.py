"""One batch split over devices (batch-sharded replicas): the shard arithmetic
of the C ABI (specv_shard_bounds, host-only), and the benchmark's multi-rank
path -- one global batch cut into contiguous shards by rank, each shard
verified on its own, the outputs gathered back in order -- run as two gloo
ranks on the CPU with the oracle standing in for each rank's GPU.

Sequences are independent (SD explainer, "批量投机（Batched Speculation）"), so
the gathered outputs must equal those of the whole batch verified at once.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402
import speculative_decoding_verification_specv_gb300 as specv  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    return specv.load(build_if_missing=True)


@pytest.mark.parametrize("B", [0, 1, 2, 7, 64, 255, 256, 1000003])
@pytest.mark.parametrize("G", [1, 2, 3, 8, 64])
def test_shards_partition_the_batch(lib, B, G):
    bounds = [specv.shard_bounds(B, G, g) for g in range(G)]
    assert bounds[0][0] == 0 and bounds[-1][1] == B
    sizes = []
    for g, (lo, hi) in enumerate(bounds):
        assert lo <= hi
        if g:
            assert lo == bounds[g - 1][1]  # contiguous and in order
        sizes.append(hi - lo)
    assert max(sizes) - min(sizes) <= 1
    assert sum(1 for n in sizes if n == 0) == max(0, G - B)


def test_shard_bounds_rejects_bad_arguments(lib):
    import ctypes
    lo, hi = ctypes.c_int64(0), ctypes.c_int64(0)
    for B, G, g in [(-1, 2, 0), (4, 0, 0), (4, 65, 0), (4, 2, 2), (4, 2, -1)]:
        assert specv.raw_call("specv_shard_bounds", B, G, g, ctypes.byref(lo),
                              ctypes.byref(hi)) == 1
    assert specv.raw_call("specv_shard_bounds", 4, 2, 0, None, ctypes.byref(hi)) == 1


def test_sharded_entry_point_validates(lib):
    fake = 16
    import ctypes
    devs = (ctypes.c_int32 * 2)(0, 0)
    args = [fake] * 6 + [4, 2, 8, 0, 0, fake, fake]
    # n_shards outside 1..64, a NULL device list, a NULL input: refused before any device work
    assert specv.raw_call("specv_verify_sharded_host", *args, 0, devs) == 1
    assert specv.raw_call("specv_verify_sharded_host", *args, 65, devs) == 1
    assert specv.raw_call("specv_verify_sharded_host", *args, 2, None) == 1
    bad = list(args)
    bad[0] = None
    assert specv.raw_call("specv_verify_sharded_host", *bad, 2, devs) == 1
    bad = list(args)
    bad[6] = 0  # B = 0
    assert specv.raw_call("specv_verify_sharded_host", *bad, 2, devs) == 1


def test_global_batch_slices_concatenate_to_the_global_batch():
    w = workloads.WORKLOADS[1].scaled(B=3)
    full = bench.global_batch_slice(w, 3, 0, 9, "cpu")
    assert full["target_logits"].shape[0] == 9
    for k in range(3):  # sub-batch j is the workload drawn with seed offset j
        xj = workloads.make_inputs(w, "cpu", seed_offset=k)
        for key in xj:
            assert torch.equal(full[key][3 * k:3 * k + 3], xj[key])
    for lo, hi in [(0, 4), (4, 9), (2, 7), (5, 5), (8, 9)]:
        part = bench.global_batch_slice(w, 3, lo, hi, "cpu")
        for key in full:
            assert torch.equal(part[key], full[key][lo:hi])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, B, out_path):
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        w = workloads.WORKLOADS[1].scaled(B=B)
        lo, hi = specv.shard_bounds(B, ws, rank)
        x = bench.global_batch_slice(w, 1, lo, hi, "cpu")  # this rank's shard of one batch
        if hi > lo:
            r = oracle.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                              x["u_accept"], x["u_resample"], x["lam"], threads=1)
            tok, n = r.tokens, r.n_accepted
        else:
            tok = np.zeros((0, w.K + 1), np.int32)
            n = np.zeros((0,), np.int32)
        tok_all, n_all = bench.gather_shards(tok, n, ws)
        if rank == 0:
            np.savez(out_path, tok=tok_all, n=n_all)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("B", [7, 1], ids=["uneven", "fewer-sequences-than-ranks"])
def test_two_gloo_ranks_shard_and_reassemble(tmp_path, lib, B):
    import oracle
    ws = 2
    out = str(tmp_path / "gathered.npz")
    mp.start_processes(_rank_main, args=(ws, _free_port(), B, out), nprocs=ws, join=True,
                       start_method="spawn")
    got = np.load(out)
    w = workloads.WORKLOADS[1].scaled(B=B)
    x = workloads.make_inputs(w, "cpu")
    ref = oracle.verify(x["target_logits"], x["draft_logits"], x["draft_tokens"], x["u_accept"],
                        x["u_resample"], x["lam"])
    np.testing.assert_array_equal(got["tok"], ref.tokens)
    np.testing.assert_array_equal(got["n"], ref.n_accepted)
