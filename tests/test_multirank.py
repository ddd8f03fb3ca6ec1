"""The benchmark's multi-rank path on CPU (gloo, world size 2).

Every rank runs an independent replica of the workload (the attention of independent
sequences needs no exchange); the harness only synchronises timing: a barrier around
the timed region and the max of the per-rank step times.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    hz = bench.Harness("gloo")
    try:
        assert hz.world == world and hz.rank == rank
        hz.barrier()
        layers = bench.shard_layers(16, world, rank)
        t = hz.max(1.5 + rank)            # per-rank step times 1.5 and 2.5 ms
        out[rank] = (t, len(layers))
        hz.barrier()
    finally:
        hz.close()


def test_two_ranks_replicate_and_take_max_time():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (2.5, 16)


def test_single_rank_harness_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    hz = bench.Harness("gloo")
    assert hz.world == 1 and hz.max(3.0) == 3.0
    hz.barrier()
    hz.close()
    assert not dist.is_initialized()


def test_workload_flop_and_byte_counts():
    from causal_gqa_flash_attention_gb300 import synthetic
    w = synthetic.WORKLOADS[2]
    P = 512 * 513 // 2
    assert w.flops() == 14 * 64 * P * 16 * 12
    assert abs(w.flops() / 1e9 - 22.59) < 0.01
    cb = w.compulsory_bytes()
    # forward reads Q, K, V and writes O and LSE
    assert cb["fwd"] == 2 * 16 * 512 * 12 * 64 * 2 + 2 * 16 * 512 * 4 * 64 * 2 + 16 * 12 * 512 * 4
