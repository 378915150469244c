"""Multi-rank sharding logic on CPU (gloo, world size 2): each rank takes its
row shard of a packed matrix and the oracle computes the shard's outputs;
gathering (axis 1) or summing (axis 0) across ranks must reproduce the
single-rank result."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from trellis_coded_weight_gb300 import inputs, shard


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    k, L, T = 3, 16, 256
    # axis 1: rows are outputs -> all_gather of the shard outputs
    codes, scales, x = inputs.make_linear(37, 512, k, 2, seed_codes=5)
    c, s, (a, b) = shard.shard_codes(codes, scales, rank, world)
    ref, _ = oracle.matvec_axis1(c, s, x, k, L, T)
    parts = [None] * world
    dist.all_gather_object(parts, (a, b, ref))
    # axis 0: rows are inputs -> all_reduce of the partial sums
    codes0, scales0, x0 = inputs.make_linear(41, 512, k, 2, seed_codes=6, sigma=0.5, x_len=41)
    c0, s0, (a0, b0) = shard.shard_codes(codes0, scales0, rank, world)
    part, _ = oracle.matvec_axis0(c0, s0, np.ascontiguousarray(x0[:, a0:b0]), k, L, T)
    t = torch.from_numpy(part)
    dist.all_reduce(t)
    if rank == 0:
        q.put((parts, t.numpy()))
    dist.barrier()
    dist.destroy_process_group()


def test_row_range_partitions():
    for rows in (1, 7, 17408):
        for world in (1, 2, 3, 8):
            spans = [shard.row_range(rows, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [e - s for s, e in spans]
            assert max(sizes) - min(sizes) <= 1


def test_two_rank_shards_reproduce_single_rank(oracle_mod):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    parts, red0 = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    k, L, T = 3, 16, 256
    codes, scales, x = inputs.make_linear(37, 512, k, 2, seed_codes=5)
    full, _ = oracle_mod.matvec_axis1(codes, scales, x, k, L, T)
    got = np.zeros_like(full)
    for a, b, ref in parts:
        got[:, a:b] = ref
    assert np.array_equal(got, full)
    codes0, scales0, x0 = inputs.make_linear(41, 512, k, 2, seed_codes=6, sigma=0.5, x_len=41)
    full0, ab0 = oracle_mod.matvec_axis0(codes0, scales0, x0, k, L, T)
    assert np.allclose(red0, full0, rtol=0, atol=1e-12 * ab0.max())
