"""Orchestration of whole indexer steps over the C ABI (no arithmetic of its own).

``fill_paged_cache`` inserts a workload's k into a device cache through
``idx_k_quant_and_cache``; ``DecodeStep`` owns the device buffers of one dense
decode step (k insert of the new tokens, paged logits, top-k, slot conversion)
``HierarchicalStep`` those of one V4.1 consumer-layer step (candidate
expansion, sparse logits, sparse top-k with remap, slot conversion), and
``DcpDecodeStep`` those of one rank of a context-parallel decode step (scoring
of the rank's own shard, local top-k with scores, one exchange, merge). Buffers
are allocated once at construction; ``run`` allocates nothing but the exchange's
receive lists. ``kv="mxfp4"`` selects the MXFP4 indexer cache (the V4.1 format)
for the cache fill and the decode and hierarchical steps.
"""

from __future__ import annotations

import numpy as np
import torch

from . import (idx_dcp_topk_merge, idx_expand_candidates, idx_k_quant_and_cache, idx_k_quant_and_cache_mxfp4,
               idx_paged_mqa_logits_decode, idx_paged_mqa_logits_decode_mxfp4, idx_req_to_global_slots,
               idx_sparse_topk_remap, idx_topk, idx_workspace_bytes)
from . import workloads as W


def _workspace(op: str, rows: int, ld: int, k: int, device) -> torch.Tensor | None:
    """The selection workspace (first-digit histograms, zero between steps), or None
    where the selection of these rows would not read it."""
    with torch.cuda.device(torch.device(device)):
        nbytes = idx_workspace_bytes(op, rows, ld, k)
    return torch.zeros((nbytes // 4,), dtype=torch.int32, device=device).view(rows, 1024) if nbytes else None


def _insert(kv: str):
    return idx_k_quant_and_cache_mxfp4 if kv == "mxfp4" else idx_k_quant_and_cache


def _decode_logits(kv: str):
    return idx_paged_mqa_logits_decode_mxfp4 if kv == "mxfp4" else idx_paged_mqa_logits_decode


def cache_block_stride(kv: str = "fp8", block_size: int = W.BLOCK_SIZE) -> int:
    """Bytes per block of the cache format (512-byte aligned): 8704 (e4m3) or 4608 (MXFP4) for 64 tokens."""
    return W.mxfp4_block_stride_bytes(block_size) if kv == "mxfp4" else W.block_stride_bytes(block_size)


def fill_paged_cache(pool: W.PagedPool, seed: int, cache: torch.Tensor, device_k: bool = False,
                     chunk_tokens: int = 1 << 21, stream=None, kv: str = "fp8") -> None:
    """Quantise and insert every request's k into ``cache`` through the cache format's insert.

    k comes from ``workloads.make_k`` (host generator) or, with ``device_k``,
    from ``workloads.make_k_device`` (for pools too large to draw on the host).
    """
    idx_k_quant_and_cache = _insert(kv)
    dev = cache.device
    if device_k:
        for b in range(len(pool.ctx_lens)):
            L = int(pool.ctx_lens[b])
            k = W.make_k_device(seed, b, L, dev)
            s = torch.from_numpy(pool.slot_mapping(b)).to(dev)
            idx_k_quant_and_cache(k, s, cache, pool.block_size, stream=stream)
        torch.cuda.current_stream(dev).synchronize()
        return
    pend_k, pend_s, n = [], [], 0

    def flush():
        nonlocal pend_k, pend_s, n
        if not pend_k:
            return
        k = torch.from_numpy(np.concatenate(pend_k).view(np.int16)).to(dev)
        s = torch.from_numpy(np.concatenate(pend_s)).to(dev)
        idx_k_quant_and_cache(k.view(torch.bfloat16), s, cache, pool.block_size, stream=stream)
        torch.cuda.current_stream(dev).synchronize()
        pend_k, pend_s, n = [], [], 0

    for b in range(len(pool.ctx_lens)):
        L = int(pool.ctx_lens[b])
        pend_k.append(W.make_k(seed, b, L))
        pend_s.append(pool.slot_mapping(b))
        n += L
        if n >= chunk_tokens:
            flush()
    flush()


class DecodeStep:
    """One dense decode step of the indexer for a fixed batch shape."""

    def __init__(self, batch: int, max_ctx: int, topk: int = W.TOPK, next_n: int = 1,
                 block_size: int = W.BLOCK_SIZE, block_span: int | None = None, device="cuda",
                 kv: str = "fp8"):
        rows = batch * next_n
        self.batch, self.next_n, self.topk = batch, next_n, topk
        self.insert, self.logits_call = _insert(kv), _decode_logits(kv)
        self.block_size = block_size
        self.block_span = block_size if block_span is None else block_span
        ld = (max_ctx + 63) // 64 * 64   # 256-byte aligned rows: vector loads in the selection
        self.logits = torch.empty((rows, ld), dtype=torch.float32, device=device)
        self.local = torch.empty((rows, topk), dtype=torch.int32, device=device)
        self.slots = torch.empty((rows, topk), dtype=torch.int32, device=device)
        self.row_ke = torch.empty(rows, dtype=torch.int32, device=device)
        # No selection workspace: without the first-digit histogram the scoring
        # kernel keeps five k stages in flight instead of four, which saves more
        # than the selection's own first-digit sweep costs (128K decode step
        # 282.3 -> 281.3 us, 64 x U[8K,32K] 49.9 -> 49.4 us on a GB300).
        self.ws = None

    def run(self, q, w, cache, block_table, ctx_lens, new_k=None, new_slots=None, row_ke=None,
            stream=None):
        """Insert new k (optional), score, select, convert; returns the slot table."""
        if new_k is not None:
            self.insert(new_k, new_slots, cache, self.block_size, stream=stream)
        self.logits_call(q, w, cache, self.block_size, block_table, ctx_lens, self.logits,
                         next_n=self.next_n, ws=self.ws, stream=stream)
        ke = ctx_lens if (row_ke is None and self.next_n == 1) else row_ke
        # selection with the slot conversion fused into its output pass
        idx_topk(self.logits, None, ke, self.topk, self.local, ws=self.ws, stream=stream,
                 slots=self.slots, block_table=block_table, block_size=self.block_size,
                 block_span=self.block_span,
                 row_to_req=None if self.next_n == 1 else self._row_to_req(ctx_lens))
        return self.slots

    def _row_to_req(self, ctx_lens):
        if not hasattr(self, "_r2r"):
            self._r2r = torch.arange(self.batch, dtype=torch.int32, device=ctx_lens.device)
            self._r2r = self._r2r.repeat_interleave(self.next_n)
        return self._r2r


class HierarchicalStep:
    """One V4.1 decode step for the consumer layers: expand once, then score, select + remap, slots.

    [V41] 功能与动机 / 实现拆解 item 2: the candidate expansion (and the schedule)
    is done once per step and shared by every consumer layer of that step;
    ``expand`` fills ``sparse_idx`` / ``end`` and ``score`` runs one layer on
    them (any number of times, the expansion buffers are only read). With
    ``next_n > 1`` (multi-token prediction) every request has ``next_n`` query
    rows, row ``r`` belonging to request ``r // next_n``, each with its own
    causal limit (``row_ke``) and candidates.
    """

    def __init__(self, rows: int, n_cand: int, cand_block_size: int = 64, sbk: int = 64,
                 topk: int = W.TOPK, block_size: int = W.BLOCK_SIZE, device="cuda", next_n: int = 1,
                 kv: str = "fp8"):
        R = cand_block_size // sbk
        self.logits_call = _decode_logits(kv)
        self.cand_block_size, self.sbk, self.topk, self.block_size = cand_block_size, sbk, topk, block_size
        self.next_n = next_n
        self.sparse_idx = torch.empty((rows, n_cand * R), dtype=torch.int32, device=device)
        self.end = torch.empty(rows, dtype=torch.int32, device=device)
        self.logits = torch.empty((rows, n_cand * R * sbk), dtype=torch.bfloat16, device=device)
        self.cols = torch.empty((rows, topk), dtype=torch.int32, device=device)
        self.positions = torch.empty((rows, topk), dtype=torch.int32, device=device)
        self.slots = torch.empty((rows, topk), dtype=torch.int32, device=device)
        self.ws = _workspace("sparse_topk_remap", rows, n_cand * R * sbk, topk, device)
        self.row_to_req = (None if next_n == 1 else
                           torch.arange(rows // next_n, dtype=torch.int32, device=device).repeat_interleave(next_n))

    def expand(self, cand, ctx_lens, row_ke=None, stream=None):
        """Once per step. ``row_ke`` (int32 [rows]) is required when ``next_n > 1``."""
        ke = ctx_lens if row_ke is None else row_ke
        idx_expand_candidates(cand, None, ke, self.cand_block_size, self.sbk, self.sparse_idx, self.end,
                              stream=stream)

    def score(self, q, w, cache, block_table, ctx_lens, stream=None):
        """One consumer layer on the current expansion; returns the slot table."""
        self.logits_call(q, w, cache, self.block_size, block_table, ctx_lens, self.logits,
                         next_n=self.next_n, sparse_idx=self.sparse_idx, end=self.end,
                         sbk=self.sbk, ws=self.ws, stream=stream)
        idx_sparse_topk_remap(self.logits, self.end, self.sparse_idx, None, self.sbk, self.topk,
                              self.positions, col_scratch=self.cols, ws=self.ws, stream=stream,
                              slots=self.slots, block_table=block_table, block_size=self.block_size,
                              block_span=self.block_size, row_to_req=self.row_to_req)
        return self.slots

    def run(self, q, w, cache, block_table, ctx_lens, cand, row_ke=None, stream=None):
        self.expand(cand, ctx_lens, row_ke, stream=stream)
        return self.score(q, w, cache, block_table, ctx_lens, stream=stream)


def exchange_candidates(vals: torch.Tensor, idx: torch.Tensor, group=None):
    """The one exchange of context-parallel decode: every rank's local top-k.

    [DSA] 几个容易踩的点: ranks that each hold a shard of a long context send
    each other only their local (score, index) lists, never the score matrix.
    ``vals`` float32 / ``idx`` int32 ``[rows, k_local]`` on each rank become
    ``[rows, world * k_local]`` on every rank, rank after rank along the row, the
    candidate layout ``idx_dcp_topk_merge`` reads. Any backend whose tensors
    these are will do (gloo with host tensors, NCCL with device tensors).
    """
    import torch.distributed as dist

    world = dist.get_world_size(group)
    gv = [torch.empty_like(vals) for _ in range(world)]
    gi = [torch.empty_like(idx) for _ in range(world)]
    dist.all_gather(gv, vals.contiguous(), group=group)
    dist.all_gather(gi, idx.contiguous(), group=group)
    return torch.cat(gv, dim=1), torch.cat(gi, dim=1)


class DcpDecodeStep:
    """One rank of a context-parallel decode step.

    The rank's paged cache holds only its shard of every request's context
    (``ctx_lens`` are shard lengths). ``select_local`` scores that shard and keeps
    its top-k with scores; ``merge`` turns every rank's lists, gathered rank after
    rank, into global top-k positions; ``run`` chains the two around
    ``exchange_candidates``. ``shard_offset`` / ``pos_stride`` give each rank's
    global positions (see ``idx_dcp_topk_merge``): per-request first positions of
    contiguous shards ([rows, world], stride 1), or ``arange(world)`` with stride
    ``world`` when tokens are dealt round-robin.
    """

    def __init__(self, batch: int, max_shard_ctx: int, world: int, topk: int = W.TOPK,
                 block_size: int = W.BLOCK_SIZE, device="cuda"):
        self.topk, self.block_size, self.world = topk, block_size, world
        ld = (max_shard_ctx + 63) // 64 * 64
        self.logits = torch.empty((batch, ld), dtype=torch.float32, device=device)
        self.cand_vals = torch.empty((batch, topk), dtype=torch.float32, device=device)
        self.cand_idx = torch.empty((batch, topk), dtype=torch.int32, device=device)
        self.positions = torch.empty((batch, topk), dtype=torch.int32, device=device)
        self.scores = torch.empty((batch, topk), dtype=torch.float32, device=device)
        self.ws = _workspace("topk", batch, ld, topk, device)

    def select_local(self, q, w, cache, block_table, ctx_lens, stream=None):
        idx_paged_mqa_logits_decode(q, w, cache, self.block_size, block_table, ctx_lens, self.logits,
                                    ws=self.ws, stream=stream)
        idx_topk(self.logits, None, ctx_lens, self.topk, self.cand_idx, vals=self.cand_vals, ws=self.ws,
                 stream=stream)
        return self.cand_vals, self.cand_idx

    def merge(self, all_vals, all_idx, shard_offset, pos_stride: int = 1, stream=None):
        idx_dcp_topk_merge(all_vals, all_idx, shard_offset, self.topk, self.topk, self.positions,
                           vals=self.scores, pos_stride=pos_stride, stream=stream)
        return self.positions

    def run(self, q, w, cache, block_table, ctx_lens, shard_offset, pos_stride: int = 1, group=None):
        """All three stages on torch's current stream, which the exchange also orders on."""
        self.select_local(q, w, cache, block_table, ctx_lens)
        all_vals, all_idx = exchange_candidates(self.cand_vals, self.cand_idx, group)
        return self.merge(all_vals, all_idx, shard_offset, pos_stride)
