"""The multi-GPU path on the host: two `gloo` ranks on CPU.

Rows are independent, so N GPUs split a batch by rows with no exchange;
the job's time is the slowest rank's and its throughput counts every rank's
bytes.  The ranks here run the oracle on their shards; the gathered result
must equal one unsharded run, and the helpers the benchmark uses for the
max-over-ranks time and the aggregate value must agree with the definition.
"""
import os
import socket

import numpy as np
import pytest

import bench
import synth

torch = pytest.importorskip("torch")


def test_shard_rows_cover_every_row_once():
    for rows in (0, 1, 7, 262143, 16384):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_rows(rows, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_aggregate_value():
    assert bench.aggregate_gbps(1e9, 10, 1, 2.0) == pytest.approx(5.0)
    assert bench.aggregate_gbps(1e9, 10, 4, 2.0) == pytest.approx(20.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    import oracle
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    rows, H = 37, 96
    x = synth.normal_bf16(31, 0, rows * H).reshape(rows, H)
    w = synth.normal_bf16(31, 2, H, 1.0, 0.1)
    r0, r1 = bench.shard_rows(rows, world, rank)
    y = oracle.rms_norm(x[r0:r1], w, 1e-6)
    # gather the shards (padded to equal size) on every rank
    n = -(-rows // world)
    pad = np.zeros((n, H), np.int32)
    pad[: r1 - r0] = y.astype(np.int32)
    parts = [torch.zeros((n, H), dtype=torch.int32) for _ in range(world)]
    dist.all_gather(parts, torch.from_numpy(pad))
    full = np.concatenate([p.numpy()[: b - a] for p, (a, b) in
                           zip(parts, [bench.shard_rows(rows, world, r) for r in range(world)])])
    # the job's time is the slowest rank's
    t = bench.max_over_ranks(0.25 + rank, world)
    if rank == 0:
        np.save(os.path.join(out_dir, "gathered.npy"), full.astype(np.uint16))
        np.save(os.path.join(out_dir, "tmax.npy"), np.array([t]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows(tmp_path):
    import torch.multiprocessing as mp
    import oracle
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows, H = 37, 96
    x = synth.normal_bf16(31, 0, rows * H).reshape(rows, H)
    w = synth.normal_bf16(31, 2, H, 1.0, 0.1)
    assert np.array_equal(np.load(tmp_path / "gathered.npy"), oracle.rms_norm(x, w, 1e-6))
    assert float(np.load(tmp_path / "tmax.npy")[0]) == pytest.approx(1.25)
