"""GB300-native FP8 lightning indexer: Python binding over the C ABI of ``libidx.so``.

Every function here only marshals arguments (torch tensors -> device pointers,
row strides, the current CUDA stream) and calls the entry point of the same
name declared in ``include/idx.h``; every step of the computation runs in the
library's CUDA kernels. A non-OK status raises :class:`IdxError` with the
library's message. The library must have been built (``build.build_library``);
importing the binding without it works, calling it raises.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib

__all__ = [
    "IdxError", "idx_k_quant_and_cache", "idx_k_quant_and_cache_mxfp4", "idx_gather_k", "idx_gather_k_mxfp4",
    "idx_mqa_logits_prefill", "idx_mqa_logits_prefill_mxfp4", "idx_paged_mqa_logits_decode", "idx_paged_mqa_logits_decode_mxfp4", "idx_topk", "idx_expand_candidates", "idx_sparse_topk_remap",
    "idx_req_to_global_slots", "idx_dcp_topk_merge", "idx_q_rope_quant", "idx_block_span",
    "idx_workspace_bytes", "idx_device_error", "library",
]


class IdxError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: status {status}: {message}")
        self.status = status


def library() -> ctypes.CDLL:
    return _lib.load()


def _check(fn: str, status: int) -> None:
    if status != _lib.IDX_OK:
        msg = library().idx_last_error().decode(errors="replace")
        raise IdxError(fn, status, msg)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return _lib.IDX_F32
    if t.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return _lib.IDX_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _rows(t: torch.Tensor) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("2-D tensor with unit column stride expected")
    return t.stride(0)


def idx_k_quant_and_cache(k, slot_mapping, cache, block_size, ue8m0=False, stream=None):
    """k [n, 128] bf16/f32, slot_mapping int64 [n], cache uint8 [num_blocks, block_stride].

    ``ue8m0``: power-of-two scales (the UE8M0 scale format) instead of amax / 448.
    """
    ld_k = _rows(k)
    _check("idx_k_quant_and_cache", library().idx_k_quant_and_cache(
        _ptr(k), _dtype_code(k), ld_k, k.shape[0], _ptr(slot_mapping), _ptr(cache),
        cache.shape[0], block_size, cache.stride(0),
        _lib.IDX_SCALE_UE8M0 if ue8m0 else _lib.IDX_SCALE_FP32, _stream(stream)))


def idx_k_quant_and_cache_mxfp4(k, slot_mapping, cache, block_size, stream=None):
    """k [n, 128] bf16/f32 -> MXFP4 cache uint8 [num_blocks, block_stride] (68 bytes per token)."""
    _check("idx_k_quant_and_cache_mxfp4", library().idx_k_quant_and_cache_mxfp4(
        _ptr(k), _dtype_code(k), _rows(k), k.shape[0], _ptr(slot_mapping), _ptr(cache),
        cache.shape[0], block_size, cache.stride(0), _stream(stream)))


def idx_gather_k(cache, block_size, block_table_row, n_tok, k8_out, kscale_out, stream=None):
    """Copy n_tok tokens of one request (block_table_row int32) into k8_out [n, 128] / kscale_out [n]."""
    _check("idx_gather_k", library().idx_gather_k(
        _ptr(cache), block_size, cache.stride(0), _ptr(block_table_row), n_tok, _ptr(k8_out),
        _ptr(kscale_out), _stream(stream)))


def idx_gather_k_mxfp4(cache, block_size, block_table_row, n_tok, codes_out, scales_out, stream=None):
    """Copy n_tok tokens of one request out of an MXFP4 cache into codes_out uint8 [n, 64] /
    scales_out int32 [n] (the words of four E8M0 codes)."""
    _check("idx_gather_k_mxfp4", library().idx_gather_k_mxfp4(
        _ptr(cache), block_size, cache.stride(0), _ptr(block_table_row), n_tok, _ptr(codes_out),
        _ptr(scales_out), _stream(stream)))


def _q_stride(q: torch.Tensor) -> int:
    if q.dim() != 3 or q.shape[1:] != (64, 128) or q.stride(2) != 1 or q.stride(1) != 128:
        raise ValueError("q must be uint8 [rows, 64, 128] with contiguous heads")
    return q.stride(0)


def idx_mqa_logits_prefill(q, w, k8, kscale, row_ks, row_ke, logits, sparse_idx=None, end=None,
                           sbk=0, n_si=None, ws=None, stream=None):
    """Dense (sparse_idx None) or sparse prefill logits; see include/idx.h."""
    ld_si = sparse_idx.stride(0) if sparse_idx is not None else 0
    if n_si is None:
        n_si = sparse_idx.shape[1] if sparse_idx is not None else 0
    _check("idx_mqa_logits_prefill", library().idx_mqa_logits_prefill(
        _ptr(q), _q_stride(q), _ptr(w), _dtype_code(w), _rows(w), _ptr(k8), _ptr(kscale),
        k8.shape[0], _ptr(row_ks), _ptr(row_ke), q.shape[0], _ptr(sparse_idx), ld_si, n_si,
        _ptr(end), sbk, _ptr(logits), _dtype_code(logits), _rows(logits), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def idx_mqa_logits_prefill_mxfp4(q, w, k_codes, k_scales, logits, sparse_idx, end, sbk, n_si=None, ws=None,
                                 stream=None):
    """Sparse prefill logits over gathered MXFP4 k (k_codes uint8 [S, 64], k_scales int32 [S])."""
    n_si = sparse_idx.shape[1] if n_si is None else n_si
    _check("idx_mqa_logits_prefill_mxfp4", library().idx_mqa_logits_prefill_mxfp4(
        _ptr(q), _q_stride(q), _ptr(w), _dtype_code(w), _rows(w), _ptr(k_codes), _ptr(k_scales),
        k_codes.shape[0], None, None, q.shape[0], _ptr(sparse_idx), sparse_idx.stride(0), n_si,
        _ptr(end), sbk, _ptr(logits), _dtype_code(logits), _rows(logits), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def idx_paged_mqa_logits_decode(q, w, cache, block_size, block_table, ctx_lens, logits, next_n=1,
                                sparse_idx=None, end=None, sbk=0, n_si=None, ws=None, stream=None):
    """Dense (sparse_idx None) or sparse decode logits read through the block table."""
    ld_si = sparse_idx.stride(0) if sparse_idx is not None else 0
    if n_si is None:
        n_si = sparse_idx.shape[1] if sparse_idx is not None else 0
    _check("idx_paged_mqa_logits_decode", library().idx_paged_mqa_logits_decode(
        _ptr(q), _q_stride(q), _ptr(w), _dtype_code(w), _rows(w), _ptr(cache), cache.shape[0],
        block_size, cache.stride(0), _ptr(block_table), _rows(block_table), _ptr(ctx_lens),
        ctx_lens.shape[0], next_n, _ptr(sparse_idx), ld_si, n_si, _ptr(end), sbk, _ptr(logits),
        _dtype_code(logits), _rows(logits), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def idx_paged_mqa_logits_decode_mxfp4(q, w, cache, block_size, block_table, ctx_lens, logits, next_n=1,
                                      sparse_idx=None, end=None, sbk=0, n_si=None, ws=None, stream=None):
    """idx_paged_mqa_logits_decode over an MXFP4 cache (dense next_n 1, or sparse)."""
    ld_si = sparse_idx.stride(0) if sparse_idx is not None else 0
    if n_si is None:
        n_si = sparse_idx.shape[1] if sparse_idx is not None else 0
    _check("idx_paged_mqa_logits_decode_mxfp4", library().idx_paged_mqa_logits_decode_mxfp4(
        _ptr(q), _q_stride(q), _ptr(w), _dtype_code(w), _rows(w), _ptr(cache), cache.shape[0],
        block_size, cache.stride(0), _ptr(block_table), _rows(block_table), _ptr(ctx_lens),
        ctx_lens.shape[0], next_n, _ptr(sparse_idx), ld_si, n_si, _ptr(end), sbk, _ptr(logits),
        _dtype_code(logits), _rows(logits), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def idx_topk(logits, row_ks, row_ke, k, out, vals=None, ws=None, stream=None, slots=None,
             block_table=None, block_size=None, block_span=None, row_to_req=None):
    """Per-row top-k indices (request-local), -1 filled; out int32 [rows, >= k]; optional scores.

    With ``slots`` (int32 [rows, >= k]) the slot conversion of idx_req_to_global_slots
    (``block_table``, ``block_size``, ``block_span``, ``row_to_req``) is fused into the
    selection's output pass (idx_topk_slots; no ``vals`` then)."""
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    if slots is None:
        _check("idx_topk", library().idx_topk(
            _ptr(logits), _dtype_code(logits), _rows(logits), _ptr(row_ks), _ptr(row_ke), logits.shape[0],
            k, _ptr(out), _rows(out), _ptr(vals), 0 if vals is None else _rows(vals), _ptr(ws), wsb,
            _stream(stream)))
        return
    if vals is not None:
        raise ValueError("idx_topk: the fused slot conversion has no score output")
    _check("idx_topk_slots", library().idx_topk_slots(
        _ptr(logits), _dtype_code(logits), _rows(logits), _ptr(row_ks), _ptr(row_ke), logits.shape[0],
        k, _ptr(out), _rows(out), _ptr(row_to_req), _ptr(block_table), _rows(block_table), block_size,
        block_span, _ptr(slots), _rows(slots), _ptr(ws), wsb, _stream(stream)))


def idx_q_rope_quant(q, positions, cos_sin, w, q8, w_out, softmax_scale, n_head_scale,
                     interleaved=False, stream=None):
    """Partial RoPE (dims 0-63), per-head e4m3 quantisation and folded weights.

    q [T, 64, 128] (or [T, 8192]) bf16/fp32, positions int32 [T], cos_sin fp32
    [max_pos, >= 64] (cos of the 32 pair angles, then sin), w [T, 64] bf16/fp32;
    writes q8 uint8 [T, 64, 128] and w_out [T, 64] (fp32 or bf16).
    """
    T = q.shape[0]
    q2 = q.reshape(T, -1) if q.dim() == 3 else q
    q8_2 = q8.reshape(T, -1) if q8.dim() == 3 else q8
    _check("idx_q_rope_quant", library().idx_q_rope_quant(
        _ptr(q2), _dtype_code(q2), _rows(q2) if T else 64 * 128, _ptr(positions), _ptr(cos_sin),
        _rows(cos_sin), cos_sin.shape[0], _lib.IDX_ROPE_INTERLEAVED if interleaved else _lib.IDX_ROPE_NEOX,
        _ptr(w), _dtype_code(w), _rows(w), float(softmax_scale), float(n_head_scale), T, _ptr(q8_2),
        _rows(q8_2) if T else 64 * 128, _ptr(w_out), _dtype_code(w_out), _rows(w_out), _stream(stream)))


def idx_dcp_topk_merge(cand_vals, cand_idx, shard_offset, k_local, k, out, vals=None, pos_stride=1,
                       stream=None):
    """Merge shard-local top-k candidates [rows, n_shards * k_local] into global top-k positions.

    ``shard_offset``: int32 [n_shards] shared by every row, int32 [rows, n_shards]
    per row, or None (offsets 0). Candidate index i of shard s maps to
    ``shard_offset[s] + i * pos_stride``.
    """
    if shard_offset is None:
        n_shards, ld_off = cand_vals.shape[1] // k_local, 0
    elif shard_offset.dim() == 1:
        n_shards, ld_off = shard_offset.shape[0], 0
    else:
        n_shards, ld_off = shard_offset.shape[1], _rows(shard_offset)
    _check("idx_dcp_topk_merge", library().idx_dcp_topk_merge(
        _ptr(cand_vals), _rows(cand_vals), _ptr(cand_idx), _rows(cand_idx), _ptr(shard_offset), ld_off,
        n_shards, pos_stride, k_local, cand_vals.shape[0], k, _ptr(out), _rows(out), _ptr(vals),
        0 if vals is None else _rows(vals), _stream(stream)))


def idx_expand_candidates(cand, row_ks, row_ke, cand_block_size, sbk, sparse_idx, end, stream=None):
    """cand int32 [rows, n_cand] -> sparse_idx int32 [rows, n_cand * R], end int32 [rows]."""
    _check("idx_expand_candidates", library().idx_expand_candidates(
        _ptr(cand), _rows(cand), cand.shape[0], cand.shape[1], _ptr(row_ks), _ptr(row_ke),
        cand_block_size, sbk, _ptr(sparse_idx), _rows(sparse_idx), _ptr(end), _stream(stream)))


def idx_sparse_topk_remap(sparse_logits, end, sparse_idx, row_ks, sbk, k, positions, col_scratch=None,
                          ws=None, stream=None, slots=None, block_table=None, block_size=None,
                          block_span=None, row_to_req=None):
    """Top-k over sparse columns [0, end) then column -> request-local position.

    With ``slots`` the slot conversion is fused into the output pass
    (idx_sparse_topk_remap_slots), as for idx_topk."""
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    if slots is None:
        _check("idx_sparse_topk_remap", library().idx_sparse_topk_remap(
            _ptr(sparse_logits), _dtype_code(sparse_logits), _rows(sparse_logits), _ptr(end),
            _ptr(sparse_idx), _rows(sparse_idx), _ptr(row_ks), sbk, sparse_logits.shape[0], k,
            _ptr(col_scratch), 0 if col_scratch is None else _rows(col_scratch), _ptr(positions),
            _rows(positions), _ptr(ws), wsb, _stream(stream)))
        return
    _check("idx_sparse_topk_remap_slots", library().idx_sparse_topk_remap_slots(
        _ptr(sparse_logits), _dtype_code(sparse_logits), _rows(sparse_logits), _ptr(end),
        _ptr(sparse_idx), _rows(sparse_idx), _ptr(row_ks), sbk, sparse_logits.shape[0], k,
        _ptr(col_scratch), 0 if col_scratch is None else _rows(col_scratch), _ptr(positions),
        _rows(positions), _ptr(row_to_req), _ptr(block_table), _rows(block_table), block_size,
        block_span, _ptr(slots), _rows(slots), _ptr(ws), wsb, _stream(stream)))


def idx_req_to_global_slots(local, row_to_req, block_table, block_size, block_span, slots, k=None,
                            stream=None):
    """Request-local positions int32 [rows, k] -> physical slots (block * block_span + offset)."""
    kk = local.shape[1] if k is None else k
    _check("idx_req_to_global_slots", library().idx_req_to_global_slots(
        _ptr(local), _rows(local), local.shape[0], kk, _ptr(row_to_req), _ptr(block_table),
        _rows(block_table), block_size, block_span, _ptr(slots), _rows(slots), _stream(stream)))


def idx_block_span(block_stride: int, token_stride: int) -> int:
    span = ctypes.c_int32(0)
    _check("idx_block_span", library().idx_block_span(block_stride, token_stride, ctypes.byref(span)))
    return span.value


def idx_workspace_bytes(op: str, rows: int, max_cols: int, k: int) -> int:
    return library().idx_workspace_bytes(_lib.OPS[op], rows, max_cols, k)


def idx_device_error(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a device-side failure."""
    _check("idx_device_error", library().idx_device_error(_stream(stream)))
