"""Multi-rank path on CPU: two gloo ranks split the requests, run the oracle on
their shards, and together reproduce the single-process result exactly."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from host_offload_serving_gb300.replicas import (job_throughput, max_over_ranks, replica_seed,
                                                 shard_requests)


def test_shard_requests_partitions():
    for total in (0, 1, 7, 8, 64):
        for world in (1, 2, 3, 8):
            got = [shard_requests(total, world, r) for r in range(world)]
            assert sum(c for _, c in got) == total
            pos = 0
            for first, count in got:
                assert first == pos
                pos += count
            assert max(c for _, c in got) - min(c for _, c in got) <= 1
    with pytest.raises(ValueError):
        shard_requests(4, 2, 2)


def test_throughput_and_seed():
    assert job_throughput(100, 2.0, 4) == 200.0
    assert replica_seed(5, 0) == 5 and replica_seed(5, 2) != replica_seed(5, 1)
    assert max_over_ranks(3.5) == 3.5


def _small_workload():
    from workload import get
    return get("tiny").scaled(R=5, k=16, B=32, L_ctx=512, steps=10, W_loc=4)


def _run_oracle(w, first, count):
    from oracle.coracle import OracleLayer
    from workload.traces import unit_trace
    rng = np.random.default_rng(0)
    host = rng.integers(0, 256, size=(w.R, w.P, 16), dtype=np.uint8)   # shared input
    o = OracleLayer(count, w.k, w.B, w.P, 16, host=np.ascontiguousarray(host[first:first + count]))
    o.reset()
    outs = []
    traces = [unit_trace(w, 0, r)[0] for r in range(first, first + count)]
    for t in range(w.steps):
        sel = np.stack([tr[t] for tr in traces]) if count else np.zeros((0, w.k), np.int32)
        out, e = o.resolve(sel)
        assert e == 0
        outs.append(out.copy())
    return np.stack(outs, 1) if count else np.zeros((0, w.steps, w.k), np.int32), o.lru.copy()


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _small_workload()
        first, count = shard_requests(w.R, world, rank)
        out, lru = _run_oracle(w, first, count)
        parts = [None] * world
        dist.all_gather_object(parts, (first, out, lru))
        tmax = max_over_ranks(1.0 + rank, dist)
        dist.barrier()
        if rank == 0:
            q.put((parts, tmax))
    finally:
        dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_gloo_ranks_reproduce_single_process():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    parts, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert tmax == 2.0
    w = _small_workload()
    full_out, full_lru = _run_oracle(w, 0, w.R)
    parts.sort(key=lambda x: x[0])
    np.testing.assert_array_equal(np.concatenate([p[1] for p in parts]), full_out)
    np.testing.assert_array_equal(np.concatenate([p[2] for p in parts]), full_lru)
