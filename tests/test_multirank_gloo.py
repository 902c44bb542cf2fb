"""The multi-process paths on CPU, with world-size-2 gloo process groups.

* bench.py's replica timing: the slowest rank's time, units of every rank;
* a context-parallel split of one sequence's prefix: each rank attends to its
  share of the keys (the last rank also to the draft block), the (o, lse)
  partials are all-gathered and merged by the LSE merge (LongSpec 2.C, the
  log-sum-exp fusion), which must equal the unsplit result.  The attention and
  the merge here are the oracle's; the device merge of gathered partials is
  verify_attn_combine, covered by the GPU tests;
* the importance pass split by position the same way: per-row (max, sum)
  partials all-gathered, merged, and each rank's positions normalised.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads as W

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, case):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        CASES[case](rank, world)
    finally:
        dist.destroy_process_group()


def _bench_replica_timing(rank, world):
    import bench

    dt = 0.001 * (rank + 1)  # rank 1 is the slow one
    assert bench.max_over_ranks(dt, dist) == pytest.approx(0.001 * world)
    rate = bench.whole_job_rate(1.0e6, dt, dist)
    assert rate == pytest.approx(world * 1.0e6 / (0.001 * world))
    bench.barrier(dist)


def _context_parallel_merge(rank, world):
    w = W.make_workload("tiny", seed=9, L=37, T=6, Hq=4, D=16)
    L, T = 37, 6
    q = w.q[0].numpy()
    k = w.k_cache[0, :L + T].numpy()
    v = w.v_cache[0, :L + T].numpy()
    vis = np.concatenate([np.ones((T, L), bool), oracle.draft_visibility(w)[0]], axis=1)
    # rank r takes prefix keys [r*L/world, (r+1)*L/world); the last rank adds the draft block
    a = rank * L // world
    b = (rank + 1) * L // world if rank < world - 1 else L + T
    o, lse = oracle.masked_attention(q, k[a:b], v[a:b], vis[:, a:b], w.scale)
    part = torch.from_numpy(np.concatenate([o.reshape(T * w.Hq, w.D), lse.T.reshape(T * w.Hq, 1)], axis=1))
    gathered = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(gathered, part)  # the one exchange step: (o, lse) of every rank
    g = torch.stack(gathered).numpy()
    out, lse_m = oracle.lse_merge(g[:, :, : w.D], g[:, :, w.D])
    ref, ref_lse = oracle.masked_attention(q, k, v, vis, w.scale)
    np.testing.assert_allclose(out.reshape(T, w.Hq, w.D), ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_m.reshape(T, w.Hq).T, ref_lse, rtol=0, atol=1e-12)


def _context_parallel_importance(rank, world):
    """The importance pass split by position: each rank scores its share of
    one sequence's committed keys for the listed heads, keeps per-row
    (maximum, sum of exp) partials, all-gathers those partials (the one
    exchange step, 2 floats per row and rank), merges them into each row's
    log-sum-exp and normalises its own positions; the shares concatenated are
    the unsplit importance map."""
    w = W.make_workload("sparse", seed=5, B=1, L_lo=300, L_hi=300, Hq=8, Hkv=2, D=16, T=3)
    heads = [1, 6]
    L = int(w.seqlens[0])
    q = oracle._widen(W.bf16_bits(w.q))[0]            # [T][Hq][D]
    k = oracle._widen(W.bf16_bits(w.k_cache))[0, :L]  # [L][Hkv][D]
    group = w.Hq // w.Hkv
    a, b = rank * L // world, (rank + 1) * L // world
    z = np.stack([w.scale * (q[:, h] @ k[a:b, h // group].T) for h in heads])  # [heads][T][share]
    m = z.max(axis=2)
    part = torch.from_numpy(np.stack([m, np.exp(z - m[..., None]).sum(axis=2)], axis=-1))  # [heads][T][2]
    gathered = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(gathered, part)
    g = torch.stack(gathered).numpy()  # [world][heads][T][2]
    M = g[..., 0].max(axis=0)
    lse = M + np.log((g[..., 1] * np.exp(g[..., 0] - M)).sum(axis=0))
    mine = np.exp(z - lse[..., None]).sum(axis=(0, 1))  # this rank's positions
    sizes = [(r + 1) * L // world - r * L // world for r in range(world)]
    shares = [torch.empty(n, dtype=torch.float64) for n in sizes]
    dist.all_gather(shares, torch.from_numpy(mine))
    got = torch.cat(shares).numpy()
    want = oracle.head_importance(W.bf16_bits(w.q), W.bf16_bits(w.k_cache), w.seqlens, heads, w.scale)[0, :L]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)


CASES = {"bench_replica_timing": _bench_replica_timing, "context_parallel_merge": _context_parallel_merge,
         "context_parallel_importance": _context_parallel_importance}


@pytest.mark.parametrize("case", sorted(CASES))
def test_two_gloo_ranks(case):
    oracle.build()  # once, before the ranks load it
    mp.spawn(_worker, args=(WORLD, _free_port(), case), nprocs=WORLD, join=True)
