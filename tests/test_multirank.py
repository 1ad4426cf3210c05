"""The N > 1 path on the CPU: expert-parallel shards over world_size-2 gloo
ranks.  Each rank computes its own experts' rows with the oracle (standing in
for its GPU), rank 0 gathers them, and the concatenation must equal the
single-rank result exactly: the shards need no exchange.  Also checks the
max-over-ranks timing reduction bench.py uses."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from ragged_grouped_gemm_02_gb300 import sharding
from ragged_grouped_gemm_02_gb300 import workloads as wl


def test_expert_ranges_cover_all_experts():
    for E in (1, 3, 32, 33, 64):
        for world in (1, 2, 3, 8):
            r = sharding.expert_ranges(E, world)
            assert r[0][0] == 0 and r[-1][1] == E
            assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
            sizes = [b - a for a, b in r]
            assert max(sizes) - min(sizes) <= 1


def test_shard_offsets_are_rebased():
    off = wl.offsets_from_counts([5, 0, 7, 3, 9])
    s = sharding.expert_shard(off, 2, 1)
    assert (s.expert_begin, s.expert_end) == (3, 5)
    assert (s.row_begin, s.row_end) == (12, 24)
    assert s.local_offsets.tolist() == [0, 3, 12]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, counts, K, N, seed, result_path):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = wl.make_custom(counts, K=K, N=N, seed=seed)
    shard = sharding.expert_shard(inp.offsets, world, rank)
    xb = wl.bf16_bits(inp.X)[shard.row_begin:shard.row_end]
    wb = wl.bf16_bits(inp.W)[shard.expert_begin:shard.expert_end]
    y = oracle.grouped_gemm(np.ascontiguousarray(xb), np.ascontiguousarray(wb), shard.local_offsets)
    parts = [None] * world
    dist.all_gather_object(parts, (shard.row_begin, shard.row_end, y))
    # the timing reduction: every rank reports its own time, the max wins
    t = torch.tensor([float(rank + 1)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        np.save(result_path, np.concatenate([p[2] for p in sorted(parts, key=lambda p: p[0])]))
        with open(result_path + ".max", "w") as f:
            f.write(str(float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_expert_parallel_equals_single_rank(tmp_path, oracle_mod):
    counts = [9, 0, 17, 4, 30, 1, 0, 12]
    K, N, seed = 48, 40, 41
    world = 2
    out = str(tmp_path / "gathered.npy")
    mp.spawn(_worker, args=(world, _free_port(), counts, K, N, seed, out), nprocs=world, join=True)
    inp = wl.make_custom(counts, K=K, N=N, seed=seed)
    full = oracle_mod.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    got = np.load(out)
    assert np.array_equal(got, full)
    assert float(open(out + ".max").read()) == float(world)
