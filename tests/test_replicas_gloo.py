"""The N > 1 path (replicas only) on CPU with two gloo ranks.

Each rank runs its own replica of a small step through the oracle (there is no GPU here),
the ranks agree on the slowest elapsed time with the same helper bench.py uses, and the
aggregate throughput counts every rank's units.  Replicas of the same seeded batch must
produce identical results.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_gqa_14_gb300 import replicas


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from paged_kv_gqa_14_gb300 import workloads as W

        assert replicas.rank_info() == (rank, world, rank)
        bt = W.config(1)
        q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                         bt.v_cache, bt.rope_theta)
        out = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc,
                                     bt.scale)
        dist.barrier()
        elapsed = 0.5 + rank  # stand-in timings: rank 1 is the slower replica
        slowest = replicas.max_over_ranks(elapsed, dist)
        thr = replicas.job_throughput(bt.num_tokens, world, slowest)
        np.save(os.path.join(outdir, f"out{rank}.npy"), out)
        with open(os.path.join(outdir, f"r{rank}.txt"), "w") as f:
            f.write(f"{slowest} {thr}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [open(tmp_path / f"r{r}.txt").read().split() for r in range(world)]
    for slowest, thr in res:
        assert float(slowest) == 1.5  # max over ranks, seen by every rank
        assert float(thr) == pytest.approx(world * 4 / 1.5)  # 4 new tokens per replica
    a, b = (np.load(tmp_path / f"out{r}.npy") for r in range(world))
    assert np.array_equal(a, b, equal_nan=True)


def test_single_process_helpers():
    assert replicas.max_over_ranks(3.0) == 3.0
    assert replicas.job_throughput(10, 4, 2.0) == 20.0
    with pytest.raises(ValueError):
        replicas.job_throughput(1, 1, 0.0)
