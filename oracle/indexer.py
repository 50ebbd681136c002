"""Plain CPU statement of the lightning-indexer hot path (fp64), for tests only.

Test infrastructure (see the package docstring). Page citations name the page
and its section:

* [DSA] "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解" (aiinfra.pub)
* [V41] "V4.1 索引器接入稀疏 MQA logits" (prhub.com.cn, vLLM PR #56254 review)
* [PACK] "修复 DSV4 FlashInfer 稀疏 MLA 在打包 KV 布局下的地址错误"
  (prhub.com.cn, vLLM PR #47493 review)

Shapes: H = 64 heads, D = 128 dims ([DSA] "Indexer 内部六步" step ①: 64 heads
of 128 dims for q, one shared 128-dim k). The indexer k cache stores 132 bytes
per token ([DSA] cost table and data-flow item 1): 128 e4m3 bytes plus a 4-byte
fp32 scale. Where a block keeps them is not printed; the reading used here (and
by the library) is the split block layout: block ``b`` starts at byte
``b * block_stride``; token ``i`` of the block has its 128 value bytes at
``i * 128`` and its fp32 scale at ``block_size * 128 + 4 * i``.
"""

from __future__ import annotations

import numpy as np

from .codecs import E4M3_MAX, e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode, e8m0_decode

H = 64
D = 128
TOKEN_BYTES = D + 4


# ----------------------------------------------------------------------------
# q preparation: partial RoPE, per-head quantisation, folded weights
# ----------------------------------------------------------------------------

ROPE_DIMS = 64      # [DSA] step ③: RoPE on the first 64 of the 128 dims only


def rope_pairs(interleaved: bool):
    """Indices (a, b) of the 32 rotary pairs: NeoX (i, i + 32) or interleaved (2i, 2i + 1)."""
    i = np.arange(ROPE_DIMS // 2)
    return (2 * i, 2 * i + 1) if interleaved else (i, i + ROPE_DIMS // 2)


def q_rope_quant(q, positions, cos_sin, w, softmax_scale, n_head_scale, interleaved=False):
    """Indexer q preparation, [DSA] "Indexer 内部六步" steps ③ and ④.

    ③ RoPE rotates pair i of the first 64 dims of every head by the angle whose
    cos / sin are ``cos_sin[pos, i]`` / ``cos_sin[pos, 32 + i]``; dims 64-127 pass
    through. ④ q is quantised with one scale per 128 values (one per head), and
    the weights absorb ``q_scale * softmax_scale * n_head_scale``.

    Every step that decides a byte runs in IEEE binary32 with each operation
    rounded (numpy float32 arithmetic, no fused multiply-add), the precision the
    quantised codes are defined in: ``y_a = x_a c - x_b s``, ``y_b = x_b c + x_a s``;
    ``scale = amax / 448``; ``q8 = e4m3(y / scale)`` (zero when the scale is 0);
    ``w_out = ((w * scale) * softmax_scale) * n_head_scale``. A position outside
    the table gives an all-zero head (scale 0, ``w_out = w * 0``).

    q: [T, 64, 128] values (bf16 inputs widened exactly); positions: [T];
    cos_sin: [max_pos, >= 64] float32; w: [T, 64].
    Returns (q8 uint8 [T, 64, 128], w_out float32 [T, 64], scale float32 [T, 64]).
    """
    q = np.asarray(q, dtype=np.float32).reshape(-1, H, D)
    T = q.shape[0]
    pos = np.asarray(positions, dtype=np.int64)
    cs = np.asarray(cos_sin, dtype=np.float32)
    ok = (pos >= 0) & (pos < cs.shape[0])
    c = cs[np.where(ok, pos, 0), :ROPE_DIMS // 2][:, None, :]                  # [T, 1, 32]
    s = cs[np.where(ok, pos, 0), ROPE_DIMS // 2:ROPE_DIMS][:, None, :]
    a, b = rope_pairs(interleaved)
    y = q.copy()
    xa, xb = q[:, :, a], q[:, :, b]
    y[:, :, a] = xa * c - xb * s
    y[:, :, b] = xb * c + xa * s
    y[~ok] = 0.0
    amax = np.max(np.abs(y), axis=2)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    q8 = np.zeros((T, H, D), dtype=np.uint8)
    live = scale != 0
    q8[live] = e4m3_encode(y[live] / scale[live][:, None])
    w = np.asarray(w, dtype=np.float32).reshape(T, H)
    w_out = ((w * scale) * np.float32(softmax_scale)) * np.float32(n_head_scale)
    return q8, w_out.astype(np.float32), scale


# ----------------------------------------------------------------------------
# a1: k quantisation fused with the cache insert
# ----------------------------------------------------------------------------

def ue8m0_ceil(s) -> np.ndarray:
    """The smallest power of two >= each positive binary32 ``s`` (0 stays 0).

    The UE8M0 scale format ([DSA] step ⑤'s ``scale_fmt`` option) keeps only an
    exponent: ``s = m * 2^e`` with ``m`` in [0.5, 1) is already a power of two when
    ``m == 0.5``, and otherwise rounds up to ``2^e``.
    """
    s = np.asarray(s, dtype=np.float32)
    m, e = np.frexp(s.astype(np.float64))
    up = np.where(m == 0.5, s.astype(np.float64), np.ldexp(1.0, e))
    return np.where(s == 0, 0.0, up).astype(np.float32)


def k_quant(k, ue8m0: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Per-token FP8 quantisation of k, one fp32 scale per 128 values.

    [DSA] step ⑤: k is quantised and written into the cache in one operation
    (``indexer_k_quant_and_cache(k, kv_cache, slot_mapping, quant_block_size,
    scale_fmt)``); step ④ fixes one scale per 128 elements. The scale format is
    fp32 ``amax / 448`` so the largest magnitude maps onto the e4m3 maximum.

    Steps, all in IEEE binary32 as the format fixes: ``amax = max |k_d|``;
    ``scale = amax / 448``; ``k8_d = e4m3(k_d / scale)``. A token whose scale is
    zero (all-zero k, or amax so small the division underflows) stores scale 0
    and all-zero bytes, so its logits are exactly 0. With ``ue8m0`` the binary32
    ``amax / 448`` is rounded up to a power of two (``ue8m0_ceil``) before the
    division, which is then exact.

    k: [n, 128] array of fp32 values (bf16 inputs widened exactly).
    Returns (k8 uint8 [n, 128], scale float32 [n]).
    """
    k = np.asarray(k, dtype=np.float32).reshape(-1, D)
    n = k.shape[0]
    k8 = np.zeros((n, D), dtype=np.uint8)
    scale = np.zeros(n, dtype=np.float32)
    for a in range(0, n, 4096):                   # blocks of tokens: small temporaries
        kb = k[a:a + 4096]
        amax = np.max(np.abs(kb), axis=1)
        s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
        if ue8m0:
            s = ue8m0_ceil(s)
        scale[a:a + 4096] = s
        live = s != 0
        k8[a:a + 4096][live] = e4m3_encode(kb[live] / s[live, None])
    return k8, scale


def k_quant_and_cache(k, slot_mapping, cache: np.ndarray, block_size: int, ue8m0: bool = False) -> None:
    """Quantise each token of ``k`` and write it to its slot of the paged cache.

    [DSA] step ⑤ and data-flow item 1 (132 bytes per token). ``slot_mapping[i]``
    is the physical slot ``block * block_size + offset`` of token i; a negative
    slot skips the token (the padding convention of slot-mapped inserts).

    cache: uint8 [num_blocks, block_stride], modified in place.
    """
    k8, scale = k_quant(k, ue8m0)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    for i, slot in enumerate(slots):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        cache[blk, off * D:(off + 1) * D] = k8[i]
        base = block_size * D + 4 * off
        cache[blk, base:base + 4] = np.frombuffer(scale[i:i + 1].tobytes(), dtype=np.uint8)


def cache_token(cache: np.ndarray, block_size: int, block: int, offset: int):
    """(k8 [128] uint8, scale float32) of one token in the split block layout."""
    k8 = cache[block, offset * D:(offset + 1) * D]
    base = block_size * D + 4 * offset
    scale = np.frombuffer(cache[block, base:base + 4].tobytes(), dtype=np.float32)[0]
    return k8, scale


def gather_k(cache: np.ndarray, block_size: int, block_table_row, n_tok: int):
    """Copy the first ``n_tok`` tokens of one request out of the paged cache.

    [DSA] "prefill 和 decode 用完全不同的内核": prefill works on gathered k;
    [V41] 实现拆解 and the key-symbol list name the prefill gather
    (``_gather_prefill_chunk_k``). Token ``p`` lives in block
    ``block_table_row[p // block_size]`` at offset ``p % block_size``.

    Returns (k8 uint8 [n_tok, 128], kscale float32 [n_tok]).
    """
    k8 = np.zeros((n_tok, D), dtype=np.uint8)
    ks = np.zeros(n_tok, dtype=np.float32)
    for p in range(n_tok):
        blk = int(block_table_row[p // block_size])
        k8[p], ks[p] = cache_token(cache, block_size, blk, p % block_size)
    return k8, ks


# ----------------------------------------------------------------------------
# a3 / a4: the logit definition
# ----------------------------------------------------------------------------

def _dequant_k(k8, kscale) -> np.ndarray:
    """k[s] as the cache represents it: e4m3 values times the token's fp32 scale."""
    return e4m3_decode(k8) * np.asarray(kscale, dtype=np.float64)[:, None]


def logits_row_values(q8_row, w_row, k) -> np.ndarray:
    """Scores of one query row against k given as fp64 values ``[S, 128]``.

    [DSA] step ⑥: ``sum_h weights[h] * (q[h] . k[s])``, q as raw e4m3 values
    (step ④ folds every q-side coefficient into the weights).
    """
    q = e4m3_decode(q8_row)                       # [64, 128]
    per_head = q @ np.asarray(k, dtype=np.float64).T    # [64, S]: q[t,h] . k[s]
    return np.asarray(w_row, dtype=np.float64) @ per_head


def logits_row(q8_row, w_row, k8, kscale) -> np.ndarray:
    """Scores of one query row against tokens ``k8``/``kscale`` (fp64).

    [DSA] step ⑥: ``logits[t, s] = sum_h weights[t, h] * (q[t, h] . k[s])`` with
    64 heads; step ④: every q-side coefficient (q scale, softmax scale, head
    scale) is already folded into ``weights``, so q enters as its raw e4m3
    values. k enters dequantised (value times the token's stored scale).

    q8_row [64, 128] uint8, w_row [64] values, k8 [S, 128] uint8, kscale [S].
    """
    return logits_row_values(q8_row, w_row, _dequant_k(k8, kscale))


def mqa_logits(q8, w, k8, kscale, row_ks, row_ke) -> np.ndarray:
    """Prefill logits on gathered k, with ragged causal row limits.

    Row ``t`` scores the tokens ``s`` in ``[row_ks[t], row_ke[t])``; every other
    column of the ``[T, S]`` result is ``-inf`` (not visible). Causality is
    carried by the limits: a query at position ``p`` sees ``s <= p``, so its
    ``row_ke`` is ``p + 1`` ([DSA] step ⑥; [V41] ``row_ks``/``row_ke`` in the
    rows-metadata snippet).
    """
    q8 = np.asarray(q8)
    T = q8.shape[0]
    S = np.asarray(k8).shape[0]
    out = np.full((T, S), -np.inf)
    for t in range(T):
        lo = max(int(row_ks[t]), 0)
        hi = min(int(row_ke[t]), S)
        if hi <= lo:
            continue
        out[t, lo:hi] = logits_row(q8[t], w[t], k8[lo:hi], kscale[lo:hi])
    return out


def decode_row_limit(ctx_len: int, next_n: int, j: int) -> int:
    """Number of visible tokens for query ``j`` of a request with ``next_n`` new queries.

    The request's own new tokens are already in the cache, so the context holds
    ``ctx_len`` tokens and query j (0-based among the last ``next_n``
    positions) sits at position ``ctx_len - next_n + j``; it sees everything up
    to and including itself.
    """
    return ctx_len - next_n + j + 1


def paged_decode_logits(q8, w, cache, block_size, block_table, ctx_lens, next_n=1) -> np.ndarray:
    """Decode logits read through the block table of the paged cache.

    [DSA] "prefill 和 decode 用完全不同的内核": decode does not gather, it reads the
    paged cache directly. Row ``r = b * next_n + j`` belongs to request ``b``.
    Result ``[rows, max ctx_len]``: visible columns hold the logit, columns in
    ``[limit, ctx_len)`` hold ``-inf``, columns ``>= ctx_len`` hold NaN (the
    library leaves them untouched).
    """
    ctx_lens = np.asarray(ctx_lens, dtype=np.int64)
    B = len(ctx_lens)
    rows = B * next_n
    width = int(ctx_lens.max()) if B else 0
    out = np.full((rows, width), np.nan)
    for b in range(B):
        L = int(ctx_lens[b])
        k8, ks = gather_k(cache, block_size, block_table[b], L)
        for j in range(next_n):
            r = b * next_n + j
            lim = max(min(decode_row_limit(L, next_n, j), L), 0)
            out[r, :L] = -np.inf
            if lim > 0:
                out[r, :lim] = logits_row(q8[r], w[r], k8[:lim], ks[:lim])
    return out


# ----------------------------------------------------------------------------
# a5: top-k with -1 fill
# ----------------------------------------------------------------------------

def topk_row(values, ks: int, ke: int, k: int) -> np.ndarray:
    """Top-``k`` request-local indices of one row, ``-1`` for empty slots.

    [DSA] opening section and data-flow item 2: keep the 2048 highest-scoring
    history tokens; the index table is int32 and ``-1`` marks an empty entry.
    The row's candidates are the columns ``[ks, ke)``; results are reported as
    ``s - ks``. When at most ``k`` columns are visible all of them are kept (in
    column order). Otherwise the order is a stable sort by value descending,
    then index ascending, so ties at the threshold keep the lower index. Empty
    slots sit at the tail.
    """
    values = np.asarray(values, dtype=np.float64)
    ks = int(ks)
    ke = int(ke)
    n = max(ke - ks, 0)
    out = np.full(k, -1, dtype=np.int64)
    if n <= k:
        out[:n] = np.arange(n)
        return out
    seg = values[ks:ke]
    order = np.lexsort((np.arange(n), -seg))
    out[:] = order[:k]
    return out


def topk(logits, row_ks, row_ke, k: int) -> np.ndarray:
    """``topk_row`` for every row: ``[rows, k]`` int64."""
    logits = np.asarray(logits)
    rows = logits.shape[0]
    ks = np.zeros(rows, dtype=np.int64) if row_ks is None else np.asarray(row_ks)
    return np.stack([topk_row(logits[r], ks[r], row_ke[r], k) for r in range(rows)]) if rows else \
        np.zeros((0, k), dtype=np.int64)


# ----------------------------------------------------------------------------
# context-parallel decode: merge of the ranks' local top-k lists
# ----------------------------------------------------------------------------

def dcp_topk_merge_row(cand_vals, cand_idx, shard_offset, k_local: int, k: int, pos_stride: int = 1):
    """Global top-``k`` of one row from every shard's local top-``k`` candidates.

    [DSA] 几个容易踩的点 (context parallelism): each rank selects within its
    own shard of the context and the ranks exchange only those local lists,
    never the score matrix. Candidate ``j`` of shard ``s`` (``cand_idx[s *
    k_local + j]``, shard-local, ``-1`` = empty) stands for global position
    ``shard_offset[s] + cand_idx * pos_stride`` (``shard_offset`` None: every
    offset is 0). The merged list is the candidates sorted by value descending,
    then global position ascending, cut to ``k`` and padded with ``-1`` /
    ``-inf``; empty candidates never enter it.

    Returns (positions int64 [k], values float64 [k]).
    """
    cand_vals = np.asarray(cand_vals, dtype=np.float64)
    cand_idx = np.asarray(cand_idx, dtype=np.int64)
    n_shards = len(cand_idx) // k_local if shard_offset is None else len(shard_offset)
    pos, val = [], []
    for s in range(n_shards):
        for j in range(k_local):
            i = int(cand_idx[s * k_local + j])
            if i >= 0:
                pos.append((0 if shard_offset is None else int(shard_offset[s])) + i * pos_stride)
                val.append(float(cand_vals[s * k_local + j]))
    pos = np.array(pos, dtype=np.int64)
    val = np.array(val, dtype=np.float64)
    order = np.lexsort((pos, -val))[:k]
    out_p = np.full(k, -1, dtype=np.int64)
    out_v = np.full(k, -np.inf)
    out_p[:len(order)] = pos[order]
    out_v[:len(order)] = val[order]
    return out_p, out_v


def dcp_topk_merge(cand_vals, cand_idx, shard_offset, k_local: int, k: int, pos_stride: int = 1):
    """``dcp_topk_merge_row`` for every row: (positions [rows, k], values [rows, k]).

    ``shard_offset``: one vector for every row, one row of offsets per row, or None.
    """
    rows = np.asarray(cand_idx).shape[0]
    per_row = shard_offset is not None and np.ndim(shard_offset) == 2
    res = [dcp_topk_merge_row(cand_vals[r], cand_idx[r], shard_offset[r] if per_row else shard_offset,
                              k_local, k, pos_stride) for r in range(rows)]
    if not res:
        return np.zeros((0, k), dtype=np.int64), np.zeros((0, k))
    return np.stack([a for a, _ in res]), np.stack([b for _, b in res])


# ----------------------------------------------------------------------------
# a6: request-local index -> physical slot
# ----------------------------------------------------------------------------

def packed_block_span(block_stride: int, token_stride: int) -> int:
    """Tokens per physical block of a pool: ``block_stride // token_stride``.

    [PACK] 实现拆解 item 1 and the ``_packed_block_span`` snippet: the span is
    the pool's per-block stride over its per-token stride and must divide
    exactly, else the layout is rejected.
    """
    if token_stride <= 0 or block_stride % token_stride != 0:
        raise ValueError(
            f"block stride {block_stride} is not a multiple of the token stride {token_stride}")
    return block_stride // token_stride


def req_to_global_slots(local, row_to_req, block_table, block_size: int, block_span: int) -> np.ndarray:
    """Request-local positions -> physical slots, ``-1`` preserved.

    [DSA] "几个容易踩的点": the indexer emits positions inside the request, the
    attention kernel needs paged-cache slots (``triton_convert_req_index_to_global_index``).
    [PACK] remap snippet: slot ``= (v // block_size) -> its physical block`` times
    ``block_span`` plus ``v % block_size``; negative entries stay ``-1``.
    Position ``v`` of row ``r`` uses block ``block_table[req(r), v // block_size]``.
    """
    local = np.asarray(local, dtype=np.int64)
    rows, k = local.shape
    out = np.full((rows, k), -1, dtype=np.int64)
    for r in range(rows):
        req = r if row_to_req is None else int(row_to_req[r])
        for i in range(k):
            v = int(local[r, i])
            if v < 0:
                continue
            blk = int(block_table[req][v // block_size])
            out[r, i] = blk * block_span + v % block_size
    return out


# ----------------------------------------------------------------------------
# a7: candidate expansion (V4.1 hierarchical variant)
# ----------------------------------------------------------------------------

def expand_candidates_row(cand, ks: int, ke: int, cand_block_size: int, sbk: int):
    """Flatten, filter, sort, dedupe and tail-pad one row of candidate blocks.

    [V41] 实现拆解 item 3 and the expansion snippet, in the page's order:

    1. each candidate block id ``c`` (in units of ``cand_block_size`` tokens) is
       split into ``R = cand_block_size / sbk`` sparse blocks ``c*R + j``;
    2. only sparse blocks inside the row's KV range are kept:
       ``0 <= x < ceil((ke - ks) / sbk)``; negative ids are padding;
    3. the kept ids are sorted ascending. Reading adopted here: duplicates are
       removed after sorting (the page sorts without dedupe and says duplicates
       are tolerated in production; scoring a token twice would let it enter the
       top-k twice, so the unique set is taken);
    4. ids are anchored at ``ks // sbk`` (``ks`` is required to be a multiple of
       ``sbk``);
    5. the tail is padded with the last valid id (or with the anchor when none
       is valid);
    6. ``end`` counts the valid sparse token columns: every kept block is whole
       except the last, which holds ``min(max(ke - start_of_last, 1), sbk)``.

    Returns (sparse_idx int64 [len(cand) * R], end int).
    """
    R = cand_block_size // sbk
    kv_len = max(ke - ks, 0)
    max_block = (kv_len + sbk - 1) // sbk
    kept = []
    for c in cand:
        c = int(c)
        if c < 0:
            continue
        for j in range(R):
            x = c * R + j
            if 0 <= x < max_block:
                kept.append(x)
    uniq = sorted(set(kept))
    n = len(uniq)
    base = ks // sbk
    width = len(cand) * R
    si = np.empty(width, dtype=np.int64)
    for i in range(width):
        if i < n:
            si[i] = uniq[i] + base
        else:
            si[i] = (uniq[-1] + base) if n else base
    if n == 0:
        end = 0
    else:
        last_start = uniq[-1] * sbk + ks
        end = (n - 1) * sbk + min(max(ke - last_start, 1), sbk)
    return si, end


def expand_candidates(cand, row_ks, row_ke, cand_block_size: int, sbk: int):
    """``expand_candidates_row`` over every row: (sparse_idx [rows, K*R], end [rows])."""
    cand = np.asarray(cand)
    rows = cand.shape[0]
    sis, ends = [], []
    for r in range(rows):
        ks = 0 if row_ks is None else int(row_ks[r])
        si, e = expand_candidates_row(cand[r], ks, int(row_ke[r]), cand_block_size, sbk)
        sis.append(si)
        ends.append(e)
    R = cand_block_size // sbk
    return (np.stack(sis) if rows else np.zeros((0, cand.shape[1] * R), dtype=np.int64),
            np.asarray(ends, dtype=np.int64))


# ----------------------------------------------------------------------------
# a8: sparse logits, a9: sparse top-k + remap
# ----------------------------------------------------------------------------

def sparse_column_token(si_row, c: int, sbk: int) -> int:
    """Absolute k position scored by sparse column ``c``: ``si[c // sbk] * sbk + c % sbk``."""
    return int(si_row[c // sbk]) * sbk + c % sbk


def sparse_logits_decode(q8, w, cache, block_size, block_table, row_to_req, si, end, sbk) -> np.ndarray:
    """V4.1 sparse logits read from the paged cache (decode, ``ks = 0``).

    [V41] 功能与动机 and 实现拆解 item 3: only the candidate sparse blocks are
    scored; the logit is the same weighted head sum. Column ``c`` of row ``r``
    scores token ``sparse_column_token(si[r], c)`` of request ``row_to_req[r]``;
    columns ``c >= end[r]`` are not valid and hold ``-inf``.
    Result: fp64 ``[rows, si.shape[1] * sbk]``.
    """
    si = np.asarray(si)
    rows, n_si = si.shape
    out = np.full((rows, n_si * sbk), -np.inf)
    for r in range(rows):
        req = r if row_to_req is None else int(row_to_req[r])
        e = int(end[r])
        if e <= 0:
            continue
        toks = [sparse_column_token(si[r], c, sbk) for c in range(e)]
        k8 = np.zeros((e, D), dtype=np.uint8)
        ks = np.zeros(e, dtype=np.float32)
        for i, p in enumerate(toks):
            blk = int(block_table[req][p // block_size])
            k8[i], ks[i] = cache_token(cache, block_size, blk, p % block_size)
        out[r, :e] = logits_row(q8[r], w[r], k8, ks)
    return out


def sparse_logits_prefill(q8, w, k8, kscale, si, end, sbk) -> np.ndarray:
    """V4.1 sparse logits over gathered k (prefill chunk); same column rule as decode."""
    si = np.asarray(si)
    rows, n_si = si.shape
    out = np.full((rows, n_si * sbk), -np.inf)
    for r in range(rows):
        e = int(end[r])
        if e <= 0:
            continue
        toks = np.array([sparse_column_token(si[r], c, sbk) for c in range(e)])
        out[r, :e] = logits_row(q8[r], w[r], k8[toks], kscale[toks])
    return out


def sparse_topk_remap_row(values, end: int, si_row, ks: int, sbk: int, k: int):
    """Top-``k`` over the first ``end`` sparse columns, then map columns to positions.

    [V41] 实现拆解 item 3 (``sparse_topk_remap``: top-k over the bf16 sparse
    logits, then ``_sparse_topk_remap_kernel`` maps each sparse column back to
    its request-local position) and the rows-metadata snippet (``col_indices``
    holds the column top-k). Column ``c`` maps to
    ``(si[c // sbk] - ks // sbk) * sbk + c % sbk``; ``-1`` stays ``-1``.

    Returns (cols int64 [k], positions int64 [k]).
    """
    cols = topk_row(values, 0, end, k)
    return cols, sparse_remap_columns(cols, si_row, ks, sbk)


def sparse_remap_columns(cols, si_row, ks: int, sbk: int) -> np.ndarray:
    """The remap step alone: sparse column ``c`` -> ``(si[c // sbk] - ks // sbk) * sbk + c % sbk``.

    [V41] 实现拆解 item 3 (the remap kernel after the sparse top-k); ``-1`` stays ``-1``.
    """
    cols = np.asarray(cols, dtype=np.int64)
    pos = np.full(cols.shape, -1, dtype=np.int64)
    base = ks // sbk
    for i, c in enumerate(cols):
        if c < 0:
            continue
        pos[i] = (int(si_row[c // sbk]) - base) * sbk + int(c) % sbk
    return pos


def dense_masked_topk_row(sparse_values, end: int, si_row, ks: int, ke: int, sbk: int, k: int):
    """The dense-masked selection the sparse path must reproduce.

    [V41] 功能与动机 (the old consumer scored the whole context and masked
    everything outside the candidates) and the test list (sparse and
    dense-masked ``torch.topk`` agree on the selected values): scatter the
    sparse scores to their context positions, leave every other position at
    ``-inf``, and select over ``[ks, ke)``. Returns request-local indices.
    """
    dense = np.full(max(ke, 0), -np.inf)
    for c in range(end):
        dense[sparse_column_token(si_row, c, sbk)] = sparse_values[c]
    sel = topk_row(dense, ks, ke, k)
    # a position that only carries -inf was never a candidate: it is an empty slot
    keep = [int(i) for i in sel if i >= 0 and np.isfinite(dense[ks + int(i)])]
    out = np.full(k, -1, dtype=np.int64)
    out[:len(keep)] = keep
    return out


# ----------------------------------------------------------------------------
# f2: the MXFP4 indexer cache (V4.1 path)
# ----------------------------------------------------------------------------
#
# [V41] 功能与动机 / 实现拆解 items 1-2 and 风险与影响: the V4.1 consumer layers
# read an MXFP4 indexer cache (indexer_kv_dtype "mxfp4") through an
# fp8 x fp4 sparse MQA-logits kernel. The pages print neither the layout nor
# the quantiser. Readings used here (and by the library):
#
# * the format is OCP MXFP4: the 128 dims of a token form four blocks of 32
#   consecutive elements; each element is FP4 E2M1 and each block shares one
#   E8M0 scale, so a token is 64 bytes of elements plus 4 scale bytes = 68 bytes;
# * quantisation follows the OCP MX conversion: per block, shared exponent
#   ``floor(log2(amax)) - 2`` (2 = the largest E2M1 exponent), clamped to the
#   E8M0 range [-127, 127] (an all-zero block gets -127), elements
#   ``e2m1(V / 2^shared)`` rounded to nearest even and saturated to +-6;
# * split block layout: block ``b`` at ``b * block_stride``; token ``i`` keeps its
#   64 element bytes at ``i * 64`` (dim ``d`` in byte ``d // 2``, even ``d`` in the
#   low nibble) and its four scale codes at ``block_size * 64 + 4 * i`` (byte ``j``
#   scales dims ``32 j .. 32 j + 31``);
# * q stays FP8 e4m3 with its scale folded into the weights ([DSA] step ④), so
#   a score is ``sum_h w[h] * sum_d q8[h, d] * e2m1(k[d]) * 2^(E[d // 32] - 127)``
#   with no per-token fp32 factor.

MX_BLOCK = 32
MXFP4_TOKEN_BYTES = D // 2 + D // MX_BLOCK     # 64 + 4 = 68


def mxfp4_quant(k) -> tuple[np.ndarray, np.ndarray]:
    """OCP MX conversion of k to MXFP4, one shared scale per 32 dims.

    k: [n, 128] fp32 values (bf16 inputs widened exactly).
    Returns (codes uint8 [n, 128], one e2m1 code per dim; scales uint8 [n, 4], E8M0 codes).
    Every step is exact in fp64: ``frexp`` gives ``floor(log2(amax))`` and the
    division is by a power of two.
    """
    k = np.asarray(k, dtype=np.float64).reshape(-1, D)
    n = k.shape[0]
    blocks = k.reshape(n, D // MX_BLOCK, MX_BLOCK)
    amax = np.max(np.abs(blocks), axis=2)                       # [n, 4]
    _, e = np.frexp(amax)                                       # amax = m 2^e, m in [0.5, 1): floor(log2) = e - 1
    shared = np.where(amax > 0, e - 1 - 2, -127)
    shared = np.clip(shared, -127, 127)
    q = blocks / np.ldexp(1.0, shared)[:, :, None]
    codes = e2m1_encode(q).reshape(n, D)
    return codes, (shared + 127).astype(np.uint8)


def mxfp4_values(codes, scales) -> np.ndarray:
    """k as the MXFP4 cache represents it: fp64 ``[n, 128]``."""
    codes = np.asarray(codes).reshape(-1, D)
    s = e8m0_decode(np.asarray(scales).reshape(-1, D // MX_BLOCK))
    return e2m1_decode(codes) * np.repeat(s, MX_BLOCK, axis=1)


def mxfp4_pack(codes) -> np.ndarray:
    """[n, 128] e2m1 codes -> [n, 64] bytes, dim 2i in the low nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1, D)
    return (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)


def mxfp4_unpack(packed) -> np.ndarray:
    """[n, 64] bytes -> [n, 128] e2m1 codes (inverse of ``mxfp4_pack``)."""
    b = np.asarray(packed, dtype=np.uint8).reshape(-1, D // 2)
    out = np.empty((b.shape[0], D), dtype=np.uint8)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out


def mxfp4_block_stride(block_size: int, align: int = 512) -> int:
    """Bytes per cache block: ``block_size * 68`` rounded up to ``align`` ([V41] 512 B stride rule)."""
    return (block_size * MXFP4_TOKEN_BYTES + align - 1) // align * align


def mxfp4_k_quant_and_cache(k, slot_mapping, cache: np.ndarray, block_size: int) -> None:
    """Quantise each token of ``k`` to MXFP4 and write it to its slot (negative slot: skipped).

    The MXFP4 counterpart of ``k_quant_and_cache`` ([DSA] step ⑤: quantisation
    fused with the insert), in the split block layout described above.
    """
    codes, scales = mxfp4_quant(k)
    packed = mxfp4_pack(codes)
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        cache[blk, off * (D // 2):(off + 1) * (D // 2)] = packed[i]
        base = block_size * (D // 2) + 4 * off
        cache[blk, base:base + 4] = scales[i]


def mxfp4_cache_token(cache: np.ndarray, block_size: int, block: int, offset: int):
    """(codes uint8 [128], scale codes uint8 [4]) of one token of an MXFP4 cache."""
    packed = cache[block, offset * (D // 2):(offset + 1) * (D // 2)]
    base = block_size * (D // 2) + 4 * offset
    return mxfp4_unpack(packed)[0], cache[block, base:base + 4].copy()


def mxfp4_gather_values(cache: np.ndarray, block_size: int, block_table_row, positions) -> np.ndarray:
    """fp64 k values ``[len(positions), 128]`` of request positions read through the block table.

    Position ``p`` lives in block ``block_table_row[p // block_size]`` at offset
    ``p % block_size``; the bytes are picked with array indexing, then decoded
    exactly as ``mxfp4_cache_token`` + ``mxfp4_values`` decode one token.
    """
    pos = np.asarray(list(positions), dtype=np.int64)
    blk = np.asarray(block_table_row, dtype=np.int64)[pos // block_size]
    off = pos % block_size
    half = D // 2
    packed = cache[blk[:, None], off[:, None] * half + np.arange(half)[None, :]]
    scales = cache[blk[:, None], block_size * half + 4 * off[:, None] + np.arange(4)[None, :]]
    return mxfp4_values(mxfp4_unpack(packed), scales)


def mxfp4_gather_k(cache: np.ndarray, block_size: int, block_table_row, n_tok: int):
    """Copy the first ``n_tok`` tokens of one request out of the MXFP4 cache (prefill).

    The MXFP4 twin of ``gather_k``: [V41] 实现拆解 item 2 (the builder slices the
    sparse buffers for every prefill chunk as well as for decode, and requires
    the MXFP4 indexer cache). Token ``p`` is read with ``mxfp4_cache_token`` from
    block ``block_table_row[p // block_size]`` at offset ``p % block_size``.

    Returns (packed codes uint8 [n_tok, 64], scale codes uint8 [n_tok, 4]).
    """
    packed = np.zeros((n_tok, D // 2), dtype=np.uint8)
    scales = np.zeros((n_tok, D // MX_BLOCK), dtype=np.uint8)
    for p in range(n_tok):
        codes, sc = mxfp4_cache_token(cache, block_size, int(block_table_row[p // block_size]), p % block_size)
        packed[p] = mxfp4_pack(codes[None, :])[0]
        scales[p] = sc
    return packed, scales


def sparse_logits_prefill_mxfp4(q8, w, packed, scales, si, end, sbk) -> np.ndarray:
    """``sparse_logits_prefill`` over gathered MXFP4 k (``mxfp4_gather_k``'s layout)."""
    si = np.asarray(si)
    rows, n_si = si.shape
    out = np.full((rows, n_si * sbk), -np.inf)
    for r in range(rows):
        e = int(end[r])
        if e <= 0:
            continue
        toks = np.array([sparse_column_token(si[r], c, sbk) for c in range(e)])
        kv = mxfp4_values(mxfp4_unpack(packed[toks]), scales[toks])
        out[r, :e] = logits_row_values(q8[r], w[r], kv)
    return out


def paged_decode_logits_mxfp4(q8, w, cache, block_size, block_table, ctx_lens, next_n=1) -> np.ndarray:
    """``paged_decode_logits`` over an MXFP4 cache (same row limits and fill values)."""
    ctx_lens = np.asarray(ctx_lens, dtype=np.int64)
    B = len(ctx_lens)
    out = np.full((B * next_n, int(ctx_lens.max()) if B else 0), np.nan)
    for b in range(B):
        L = int(ctx_lens[b])
        kv = mxfp4_gather_values(cache, block_size, block_table[b], range(L))
        for j in range(next_n):
            r = b * next_n + j
            lim = max(min(decode_row_limit(L, next_n, j), L), 0)
            out[r, :L] = -np.inf
            if lim > 0:
                out[r, :lim] = logits_row_values(q8[r], w[r], kv[:lim])
    return out


def sparse_logits_decode_mxfp4(q8, w, cache, block_size, block_table, row_to_req, si, end, sbk) -> np.ndarray:
    """``sparse_logits_decode`` over an MXFP4 cache: column ``c < end`` scores its mapped token."""
    si = np.asarray(si)
    rows, n_si = si.shape
    out = np.full((rows, n_si * sbk), -np.inf)
    for r in range(rows):
        req = r if row_to_req is None else int(row_to_req[r])
        e = int(end[r])
        if e <= 0:
            continue
        toks = [sparse_column_token(si[r], c, sbk) for c in range(e)]
        out[r, :e] = logits_row_values(q8[r], w[r], mxfp4_gather_values(cache, block_size, block_table[req], toks))
    return out
