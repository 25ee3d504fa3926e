"""Multi-rank path on CPU: two gloo ranks each run their shard of one forward
(with the fp64 oracle standing in for the per-rank compute, since there is no
GPU here), gather, and must reproduce the single-rank result exactly; the
benchmark's max-over-ranks timing reduction is checked the same way."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from kimi_delta_attention_gb300 import sharding


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(B, T, H, HV, K, V, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K)).astype(np.float32)
    k = rng.standard_normal((B, T, H, K)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, HV, V)).astype(np.float32)
    g = (-np.abs(rng.standard_normal((B, T, HV, K))) * 0.1).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((B, T, HV))))).astype(np.float32)
    s0 = (rng.standard_normal((B, HV, K, V)) * 0.1).astype(np.float32)
    return q, k, v, g, beta, s0


def _worker(rank, world, port, shape, q_ret):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, T, H, HV, K, V = shape
    q, k, v, g, beta, s0 = _inputs(*shape)
    sh = sharding.shard(B, H, HV, rank, world)
    parts = sharding.take(sh, q, k, v, g, beta, s0)
    o, S = oracle.forward(*parts[:5], 0.3, initial_state=parts[5], form="chunked", chunk=16, nthreads=1)
    # gather full-size results (zero outside the shard, then sum)
    o_full = np.zeros((B, T, HV, V))
    S_full = np.zeros((B, HV, K, V))
    o_full[sh.batch[0]:sh.batch[1], :, sh.heads[0]:sh.heads[1]] = o
    S_full[sh.batch[0]:sh.batch[1], sh.heads[0]:sh.heads[1]] = S
    to = torch.from_numpy(o_full)
    ts = torch.from_numpy(S_full)
    dist.all_reduce(to)
    dist.all_reduce(ts)
    # max-over-ranks step time, as the benchmark reduces it
    t = torch.tensor([1.0 + rank])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        q_ret.put((to.numpy(), ts.numpy(), float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("shape", [(2, 40, 2, 4, 8, 6),   # batch split
                                   (1, 40, 2, 8, 8, 6)])  # key-head-group split (G = 4)
def test_two_gloo_ranks_reproduce_single_rank(shape):
    import oracle
    ctx = mp.get_context("spawn")
    q_ret = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, shape, q_ret)) for r in range(2)]
    for p in procs:
        p.start()
    o, S, tmax = q_ret.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    q, k, v, g, beta, s0 = _inputs(*shape)
    o_ref, S_ref = oracle.forward(q, k, v, g, beta, 0.3, initial_state=s0, form="chunked", chunk=16)
    assert np.array_equal(o, o_ref) and np.array_equal(S, S_ref)
    assert tmax == 2.0


def test_shards_cover_every_unit_once():
    for B, H, HV, world in [(1, 32, 32, 2), (1, 8, 32, 4), (4, 32, 32, 8), (3, 2, 8, 2), (1, 1, 1, 2)]:
        seen = np.zeros((B, HV), dtype=int)
        for r in range(world):
            sh = sharding.shard(B, H, HV, r, world)
            if sh.empty:
                continue
            G = HV // H
            assert sh.heads == (sh.key_heads[0] * G, sh.key_heads[1] * G)
            seen[sh.batch[0]:sh.batch[1], sh.heads[0]:sh.heads[1]] += 1
        assert (seen == 1).all(), (B, H, HV, world)
