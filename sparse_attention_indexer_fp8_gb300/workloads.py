"""Seeded synthetic inputs for the indexer, shared by the tests and the benchmark.

This module only draws random inputs and lays them out; it holds none of the
indexer's arithmetic. The q side arrives already quantised, as the indexer
receives it (the q rope/quant producer is upstream of the scoring path): q is
drawn N(0, 1), given one fp32 scale per head (``amax / 448``) and cast to e4m3
with PyTorch's own ``float8_e4m3fn`` conversion; the per-head weights carry the
q scale and the usual ``128**-0.5 * 64**-0.5`` softmax/head factors folded in.
k is drawn N(0, 1) in bf16 and is quantised by the path under test.

All generators are CPU ``torch.Generator`` streams seeded from the workload's
seed, so every test and the benchmark see the same bytes on any machine. k of
request ``b`` has its own stream (seed, b), which lets a checker regenerate one
request's k without regenerating the whole pool.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

H = 64
D = 128
E4M3_MAX = 448.0
TOPK = 2048
BLOCK_SIZE = 64
TOKEN_BYTES = 132
BLOCK_ALIGN = 512


def block_stride_bytes(block_size: int = BLOCK_SIZE, align: int = BLOCK_ALIGN) -> int:
    """Bytes per cache block: ``block_size * 132`` rounded up to ``align`` (8704 for 64 tokens)."""
    raw = block_size * TOKEN_BYTES
    return (raw + align - 1) // align * align


MXFP4_TOKEN_BYTES = 68      # MXFP4 cache: 64 bytes of e2m1 elements + 4 E8M0 block scales


def mxfp4_block_stride_bytes(block_size: int = BLOCK_SIZE, align: int = BLOCK_ALIGN) -> int:
    """Bytes per MXFP4 cache block: ``block_size * 68`` rounded up to ``align`` (4608 for 64 tokens)."""
    raw = block_size * MXFP4_TOKEN_BYTES
    return (raw + align - 1) // align * align


def _gen(seed: int, *stream: int) -> torch.Generator:
    g = torch.Generator()
    s = int(seed)
    for x in stream:
        s = (s * 1_000_003 + int(x) + 1) % (2**62)
    g.manual_seed(s)
    return g


def make_q(seed: int, rows: int, w_bf16: bool = False):
    """(q8 uint8 [rows, 64, 128], w [rows, 64]) as the scoring kernel receives them.

    ``w`` is float32, or bf16 bit patterns (uint16) when ``w_bf16``, rounded once
    from the fp32 weights by PyTorch's cast.
    """
    g = _gen(seed, 1)
    q = torch.randn(rows, H, D, generator=g, dtype=torch.float32)
    q_scale = q.abs().amax(dim=-1) / E4M3_MAX                      # [rows, 64]
    q_scale = torch.where(q_scale > 0, q_scale, torch.ones_like(q_scale))
    q8 = (q / q_scale[..., None]).to(torch.float8_e4m3fn).view(torch.uint8)
    w_raw = torch.randn(rows, H, generator=g, dtype=torch.float32) * (1.0 / 8.0)
    w = w_raw * q_scale * (D ** -0.5) * (H ** -0.5)
    if w_bf16:
        w = w.to(torch.bfloat16).view(torch.int16)
        return q8.numpy(), w.numpy().view(np.uint16)
    return q8.numpy(), w.numpy()


def make_k(seed: int, request: int, n_tok: int) -> np.ndarray:
    """k of one request, bf16 bit patterns uint16 [n_tok, 128], N(0, 1)."""
    g = _gen(seed, 2, request)
    k = torch.randn(n_tok, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return k.view(torch.int16).numpy().view(np.uint16)


def make_k_device(seed: int, request: int, n_tok: int, device) -> torch.Tensor:
    """k of one request drawn on the device (torch's CUDA generator): bf16 [n_tok, 128], N(0, 1).

    For pools too large to draw on the host. Deterministic for a given seed,
    request and PyTorch build; a checker that needs the same k calls this
    function again and copies the result to the host.
    """
    g = torch.Generator(device=device)
    s = int(seed)
    for x in (8, request):
        s = (s * 1_000_003 + int(x) + 1) % (2**62)
    g.manual_seed(s)
    return torch.randn(n_tok, D, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_random_cache_tokens(seed: int, n_tok: int):
    """Directly drawn cache contents (k8 uint8 [n, 128] without NaN codes, kscale f32 [n])."""
    g = _gen(seed, 3)
    k8 = torch.randint(0, 254, (n_tok, D), generator=g, dtype=torch.int32)
    k8 = torch.where(k8 >= 0x7F, k8 + 1, k8)            # skip 0x7F (NaN); 0xFF is never drawn
    kscale = torch.rand(n_tok, generator=g, dtype=torch.float32) * 0.02 + 1e-3
    return k8.to(torch.uint8).numpy(), kscale.numpy()


@dataclasses.dataclass
class PagedPool:
    """A shuffled paged layout: which physical block holds each request's logical block."""

    ctx_lens: np.ndarray          # int32 [B]
    block_table: np.ndarray       # int32 [B, max_blocks]; unused entries hold 0
    num_blocks: int
    block_size: int

    def slot_mapping(self, b: int) -> np.ndarray:
        """Physical slot of every token of request b (int64 [ctx_lens[b]])."""
        L = int(self.ctx_lens[b])
        p = np.arange(L, dtype=np.int64)
        return self.block_table[b, p // self.block_size].astype(np.int64) * self.block_size + p % self.block_size


def make_pool(seed: int, ctx_lens, block_size: int = BLOCK_SIZE, extra_blocks: int = 0) -> PagedPool:
    """Assign every request's blocks to a random permutation of a pool just large enough."""
    ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
    nb = (ctx_lens.astype(np.int64) + block_size - 1) // block_size
    total = int(nb.sum()) + extra_blocks
    g = _gen(seed, 4)
    perm = torch.randperm(total, generator=g).numpy().astype(np.int32)
    max_blocks = int(nb.max()) if len(nb) else 1
    bt = np.zeros((len(ctx_lens), max(max_blocks, 1)), dtype=np.int32)
    off = 0
    for b, n in enumerate(nb):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    return PagedPool(ctx_lens, bt, total, block_size)


def uniform_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n context lengths uniform on the integers [lo, hi]."""
    g = _gen(seed, 5)
    return torch.randint(lo, hi + 1, (n,), generator=g).numpy().astype(np.int32)


def make_candidates(seed: int, rows: int, n_cand: int, n_blocks: int,
                    n_dup: int = 4, n_pad: int = 2, n_oob: int = 2) -> np.ndarray:
    """Candidate block ids a source layer publishes, as the hierarchical workload draws them.

    Per row: ``n_cand`` distinct ids in ``[0, n_blocks)``, unsorted; then
    ``n_dup`` slots are overwritten with copies of other slots, ``n_pad`` with
    -1 and ``n_oob`` with ids in ``[n_blocks, 2 * n_blocks)``.
    """
    g = _gen(seed, 6)
    out = np.zeros((rows, n_cand), dtype=np.int32)
    for r in range(rows):
        ids = torch.randperm(n_blocks, generator=g)[:n_cand].numpy().astype(np.int32)
        slots = torch.randperm(n_cand, generator=g).numpy()
        k = 0
        for _ in range(n_dup):
            src = int(slots[(k + n_dup + n_pad + n_oob) % n_cand])
            ids[slots[k]] = ids[src]
            k += 1
        for _ in range(n_pad):
            ids[slots[k]] = -1
            k += 1
        for _ in range(n_oob):
            ids[slots[k]] = n_blocks + int(torch.randint(0, n_blocks, (1,), generator=g))
            k += 1
        out[r] = ids
    return out


def make_logits(seed: int, rows: int, width: int, ties: bool = False) -> np.ndarray:
    """Random fp32 score rows for selection tests; with ``ties`` values repeat often."""
    g = _gen(seed, 7)
    x = torch.randn(rows, width, generator=g, dtype=torch.float32) * 0.1
    if ties:
        x = torch.round(x * 64.0) / 64.0
    return x.numpy()


# ----------------------------------------------------------------------------
# Named workloads (sizes from the problem statement)
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class DecodeWorkload:
    name: str
    seed: int
    pool: PagedPool
    q8: np.ndarray
    w: np.ndarray
    next_n: int = 1
    topk: int = TOPK
    block_span: int = BLOCK_SIZE

    @property
    def batch(self) -> int:
        return len(self.pool.ctx_lens)


def tiny_decode(seed: int = 1000) -> DecodeWorkload:
    """4 requests with contexts 1000/2048/3000/4096 tokens in a 256-block shuffled pool."""
    ctx = np.array([1000, 2048, 3000, 4096], dtype=np.int32)
    pool = make_pool(seed, ctx, extra_blocks=256 - 159)
    q8, w = make_q(seed, len(ctx))
    return DecodeWorkload("tiny-decode-b4", seed, pool, q8, w)


def paged_decode(seed: int = 1001, batch: int = 64) -> DecodeWorkload:
    """batch 64, contexts uniform in [8K, 32K], then slot conversion."""
    ctx = uniform_lengths(seed, batch, 8192, 32768)
    pool = make_pool(seed, ctx)
    q8, w = make_q(seed, batch)
    return DecodeWorkload("paged-decode-b64-8k32k", seed, pool, q8, w)


def long_decode(seed: int = 1003, batch: int = 128) -> DecodeWorkload:
    """batch 128, contexts uniform in [64K, 128K] (~2.2 GB of cache)."""
    ctx = uniform_lengths(seed, batch, 65536, 131072)
    pool = make_pool(seed, ctx)
    q8, w = make_q(seed, batch)
    return DecodeWorkload("long-decode-b128-64k128k", seed, pool, q8, w)


@dataclasses.dataclass
class PrefillWorkload:
    name: str
    seed: int
    S: int
    q8: np.ndarray
    w: np.ndarray            # fp32 or bf16 bits
    w_bf16: bool
    row_ks: np.ndarray
    row_ke: np.ndarray
    topk: int = TOPK


def causal_prefill(seed: int, T: int, S: int, w_bf16: bool, name: str) -> PrefillWorkload:
    """The last T positions of an S-token context: row i at position S-T+i sees [0, S-T+i]."""
    q8, w = make_q(seed, T, w_bf16=w_bf16)
    pos = np.arange(S - T, S, dtype=np.int32)
    return PrefillWorkload(name, seed, S, q8, w, w_bf16,
                           np.zeros(T, dtype=np.int32), pos + 1)


def tiny_prefill(seed: int = 1000) -> PrefillWorkload:
    return causal_prefill(seed + 50, 256, 4096, False, "tiny-prefill-256x4096")


def prefill_chunk(seed: int = 1002) -> PrefillWorkload:
    """8192 queries on a 32K context, bf16 weights."""
    return causal_prefill(seed, 8192, 32768, True, "prefill-8192x32768")


@dataclasses.dataclass
class HierarchicalWorkload:
    name: str
    seed: int
    pool: PagedPool
    q8: np.ndarray
    w: np.ndarray
    cand: np.ndarray            # int32 [B, 64] candidate block ids (64-token blocks)
    cand_block_size: int = 64
    sbk: int = 64
    topk: int = TOPK
    next_n: int = 1             # query rows per request (rows = batch * next_n)


def hierarchical(seed: int = 1004, batch: int = 128, ctx: int = 131072, n_cand: int = 64) -> HierarchicalWorkload:
    """batch 128 at 128K: 64 candidate 64-token blocks per row with duplicates, -1 and out-of-range ids."""
    lens = np.full(batch, ctx, dtype=np.int32)
    pool = make_pool(seed, lens)
    q8, w = make_q(seed, batch)
    cand = make_candidates(seed, batch, n_cand, ctx // 64)
    return HierarchicalWorkload(f"hierarchical-b{batch}-{ctx // 1024}k", seed, pool, q8, w, cand)


def hierarchical_mtp(seed: int = 1005, batch: int = 128, ctx: int = 131072, n_cand: int = 64,
                     next_n: int = 2) -> HierarchicalWorkload:
    """The hierarchical workload with next_n query rows per request, each with its own candidates."""
    lens = np.full(batch, ctx, dtype=np.int32)
    pool = make_pool(seed, lens)
    rows = batch * next_n
    q8, w = make_q(seed, rows)
    cand = make_candidates(seed, rows, n_cand, ctx // 64)
    return HierarchicalWorkload(f"hierarchical-mtp{next_n}-b{batch}-{ctx // 1024}k", seed, pool, q8, w, cand,
                                next_n=next_n)


# ----------------------------------------------------------------------------
# q preparation (partial RoPE + per-head quantisation + weight folding)
# ----------------------------------------------------------------------------

ROPE_BASE = 10000.0


def rope_cos_sin(max_pos: int, base: float = ROPE_BASE) -> np.ndarray:
    """cos / sin table [max_pos, 64] float32 of the 32 rotary pair angles pos * base^(-2i/64)."""
    i = np.arange(32, dtype=np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * base ** (-2.0 * i / 64.0)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


@dataclasses.dataclass
class QPrepWorkload:
    name: str
    seed: int
    T: int
    positions: np.ndarray   # int32 [T]
    cos_sin: np.ndarray     # float32 [max_pos, 64]
    w: np.ndarray           # float32 [T, 64]: the projection's raw head weights


def make_q_raw_device(seed: int, T: int, device) -> torch.Tensor:
    """Pre-RoPE q drawn on the device: bf16 [T, 64 * 128], N(0, 1). Deterministic per seed."""
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + 11) % (2**62))
    return torch.randn(T, H * D, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def q_prep_chunk(seed: int = 1006, T: int = 8192, ctx: int = 32768) -> QPrepWorkload:
    """The prefill chunk's queries (the last T positions of a ctx-token context)."""
    g = _gen(seed, 12)
    w = (torch.randn(T, H, generator=g, dtype=torch.float32) / 8.0).numpy()
    pos = np.arange(ctx - T, ctx, dtype=np.int32)
    return QPrepWorkload("q-prep-8192-of-32k", seed, T, pos, rope_cos_sin(ctx), w)
