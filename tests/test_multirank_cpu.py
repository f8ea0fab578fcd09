"""The multi-rank form of the benchmark on CPU: two gloo ranks, each serving its own shard of sequences.

The data path has no exchange (each rank's decode is independent); the only collective is the max over ranks of
the step time.  Here every rank builds its shard, evaluates it with the fp64 oracle (standing in for its GPU), and
the ranks reduce their times as the benchmark does."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    import oracle
    from paged_kv_cache_71_gb300 import workload as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        kw = bench.rank_workload_kwargs("tiny", rank)
        w = wl.make("tiny", **kw)
        out = oracle.paged_attention_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
        my_ms = 1.0 + rank  # a stand-in step time: rank 1 is the slower one
        job_ms = bench.max_over_ranks(my_ms, dist, "cpu")
        q.put((rank, kw.get("seed"), float(np.abs(out).sum()), job_ms,
               bench.job_throughput(world, w.num_seqs, job_ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, seed0, sum0, job0, thr0), (r1, seed1, sum1, job1, thr1) = res
    assert seed0 != seed1            # every rank serves its own sequences
    assert sum0 != sum1
    assert job0 == job1 == 2.0       # the slowest rank sets the job's step time
    from paged_kv_cache_71_gb300 import workload as wl
    n = wl.make("tiny").num_seqs
    assert thr0 == thr1 == pytest.approx(2 * n / 2.0e-3)


def test_single_process_reduction_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.rank_workload_kwargs("llama70b_mixed_fp8", 0) == {}
    assert bench.rank_workload_kwargs("llama70b_mixed_fp8", 1)["seed"] != bench.rank_workload_kwargs(
        "llama70b_mixed_bf16", 0)["seed"]
