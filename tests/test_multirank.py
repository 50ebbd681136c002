"""The multi-rank benchmark path on CPU: two gloo ranks on 127.0.0.1.

Ranks run independent batches (weak scaling) and meet only at the barrier and
the max-over-ranks reduction of the timed region; both are exercised here, and
the per-rank workloads are checked to be distinct.
"""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from sparse_attention_indexer_fp8_gb300 import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    elapsed = 10.0 + 5.0 * rank                      # each rank's own timed region
    out[rank] = bench.max_over_ranks(dist, elapsed, torch.device("cpu"))
    wl = W.paged_decode(seed=bench.rank_seed(1001, rank), batch=8)
    out[world + rank] = float(wl.pool.ctx_lens.sum())
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_gloo_ranks_share_max_time_and_own_batches():
    world = 2
    out = mp.get_context("spawn").Manager().list([0.0] * (2 * world))
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == 15.0, "every rank reports the slowest rank's time"
    assert out[2] != out[3], "ranks draw independent batches"
