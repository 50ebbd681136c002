"""Multi-rank paths on CPU: gloo ranks on 127.0.0.1.

The benchmark's ranks run independent batches (weak scaling) and meet only at
the barrier and the max-over-ranks reduction of the timed region; both are
exercised here, and the per-rank workloads are checked to be distinct.

Context-parallel decode: each rank holds a shard of every row, selects its local
top-k (the oracle stands in for the device selection), and the ranks exchange
the lists through ``exchange_candidates``; the oracle's merge of what arrives
must equal the oracle's top-k of the whole row, on every rank.
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


def _dcp_worker(rank, world, port, mode, out):
    import sys

    import numpy as np

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    from oracle import indexer as O
    from sparse_attention_indexer_fp8_gb300 import workloads as W
    from sparse_attention_indexer_fp8_gb300.pipeline import exchange_candidates

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    rows, width, k = 4, 6000, 512
    x = W.make_logits(77, rows, width, ties=True)           # every rank draws the same full rows
    lens = np.array([width, 4001, 300, 1], dtype=np.int64)
    vals = np.full((rows, k), -np.inf, dtype=np.float32)
    loc = np.full((rows, k), -1, dtype=np.int32)
    offs = np.zeros((rows, world), dtype=np.int32)
    for r in range(rows):
        n = int(lens[r])
        if mode == "contiguous":
            b = [n * i // world for i in range(world + 1)]
            offs[r] = b[:-1]
            shard = x[r, b[rank]:b[rank + 1]]
        else:
            offs[r] = np.arange(world)
            shard = x[r, rank:n:world]
        sel = O.topk_row(shard, 0, len(shard), k)
        loc[r] = sel
        vals[r, sel >= 0] = shard[sel[sel >= 0]]
    av, ai = exchange_candidates(torch.from_numpy(vals), torch.from_numpy(loc))
    av, ai = av.numpy(), ai.numpy()
    ok = av.shape == (rows, world * k) and np.array_equal(ai[:, rank * k:(rank + 1) * k], loc)
    stride = 1 if mode == "contiguous" else world
    pos, _ = O.dcp_topk_merge(av, ai, offs, k, k, stride)
    for r in range(rows):
        n = int(lens[r])
        m = min(n, k)
        ref = O.topk_row(x[r], 0, n, k)
        ok = ok and sorted(pos[r, :m].tolist()) == sorted(ref[:m].tolist()) and bool(np.all(pos[r, m:] == -1))
    out[rank] = bool(ok)
    dist.barrier()
    dist.destroy_process_group()


def _run_dcp(world, mode):
    out = mp.get_context("spawn").Manager().list([False] * world)
    mp.start_processes(_dcp_worker, args=(world, _free_port(), mode, out), nprocs=world, join=True,
                       start_method="spawn")
    return list(out)


def test_dcp_exchange_and_merge_two_ranks():
    assert _run_dcp(2, "contiguous") == [True, True]


def test_dcp_exchange_and_merge_three_ranks_round_robin():
    assert _run_dcp(3, "round_robin") == [True, True, True]
