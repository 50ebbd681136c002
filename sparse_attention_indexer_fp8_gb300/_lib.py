"""ctypes declarations of the C ABI in ``include/idx.h`` (loaded from the in-tree libidx.so)."""

from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_int = ctypes.c_int
c_ptr = ctypes.c_void_p
c_size = ctypes.c_size_t

IDX_OK = 0
IDX_F32 = 0
IDX_BF16 = 1
IDX_SCALE_FP32 = 0
IDX_SCALE_UE8M0 = 1
IDX_ROPE_NEOX = 0
IDX_ROPE_INTERLEAVED = 1

OPS = {
    "k_quant_and_cache": 1, "gather_k": 2, "mqa_logits_prefill": 3,
    "paged_mqa_logits_decode": 4, "topk": 5, "expand_candidates": 6,
    "sparse_topk_remap": 7, "req_to_global_slots": 8,
}

# name -> (restype, argtypes); one line per entry point of include/idx.h
SIGNATURES = {
    "idx_k_quant_and_cache": (c_int, [c_ptr, c_int, c_i64, c_i32, c_ptr, c_ptr, c_i32, c_i32, c_i64,
                                      c_int, c_ptr]),
    "idx_k_quant_and_cache_mxfp4": (c_int, [c_ptr, c_int, c_i64, c_i32, c_ptr, c_ptr, c_i32, c_i32, c_i64,
                                            c_ptr]),
    "idx_gather_k": (c_int, [c_ptr, c_i32, c_i64, c_ptr, c_i32, c_ptr, c_ptr, c_ptr]),
    "idx_gather_k_mxfp4": (c_int, [c_ptr, c_i32, c_i64, c_ptr, c_i32, c_ptr, c_ptr, c_ptr]),
    "idx_mqa_logits_prefill": (c_int, [c_ptr, c_i64, c_ptr, c_int, c_i64, c_ptr, c_ptr, c_i32, c_ptr,
                                       c_ptr, c_i32, c_ptr, c_i64, c_i32, c_ptr, c_i32, c_ptr, c_int,
                                       c_i64, c_ptr, c_size, c_ptr]),
    "idx_mqa_logits_prefill_mxfp4": (c_int, [c_ptr, c_i64, c_ptr, c_int, c_i64, c_ptr, c_ptr, c_i32, c_ptr,
                                       c_ptr, c_i32, c_ptr, c_i64, c_i32, c_ptr, c_i32, c_ptr, c_int,
                                       c_i64, c_ptr, c_size, c_ptr]),
    "idx_paged_mqa_logits_decode": (c_int, [c_ptr, c_i64, c_ptr, c_int, c_i64, c_ptr, c_i32, c_i32,
                                            c_i64, c_ptr, c_i64, c_ptr, c_i32, c_i32, c_ptr, c_i64,
                                            c_i32, c_ptr, c_i32, c_ptr, c_int, c_i64, c_ptr, c_size,
                                            c_ptr]),
    "idx_paged_mqa_logits_decode_mxfp4": (c_int, [c_ptr, c_i64, c_ptr, c_int, c_i64, c_ptr, c_i32, c_i32,
                                                  c_i64, c_ptr, c_i64, c_ptr, c_i32, c_i32, c_ptr, c_i64,
                                                  c_i32, c_ptr, c_i32, c_ptr, c_int, c_i64, c_ptr, c_size,
                                                  c_ptr]),
    "idx_topk": (c_int, [c_ptr, c_int, c_i64, c_ptr, c_ptr, c_i32, c_i32, c_ptr, c_i64, c_ptr, c_i64,
                         c_ptr, c_size, c_ptr]),
    "idx_q_rope_quant": (c_int, [c_ptr, c_int, c_i64, c_ptr, c_ptr, c_i64, c_i32, c_i32, c_ptr, c_int, c_i64,
                                 ctypes.c_float, ctypes.c_float, c_i32, c_ptr, c_i64, c_ptr, c_int, c_i64,
                                 c_ptr]),
    "idx_dcp_topk_merge": (c_int, [c_ptr, c_i64, c_ptr, c_i64, c_ptr, c_i64, c_i32, c_i32, c_i32, c_i32,
                                   c_i32, c_ptr, c_i64, c_ptr, c_i64, c_ptr]),
    "idx_expand_candidates": (c_int, [c_ptr, c_i64, c_i32, c_i32, c_ptr, c_ptr, c_i32, c_i32, c_ptr,
                                      c_i64, c_ptr, c_ptr]),
    "idx_sparse_topk_remap": (c_int, [c_ptr, c_int, c_i64, c_ptr, c_ptr, c_i64, c_ptr, c_i32, c_i32,
                                      c_i32, c_ptr, c_i64, c_ptr, c_i64, c_ptr, c_size, c_ptr]),
    "idx_req_to_global_slots": (c_int, [c_ptr, c_i64, c_i32, c_i32, c_ptr, c_ptr, c_i64, c_i32, c_i32,
                                        c_ptr, c_i64, c_ptr]),
    "idx_topk_slots": (c_int, [c_ptr, c_int, c_i64, c_ptr, c_ptr, c_i32, c_i32, c_ptr, c_i64, c_ptr, c_ptr,
                               c_i64, c_i32, c_i32, c_ptr, c_i64, c_ptr, c_size, c_ptr]),
    "idx_sparse_topk_remap_slots": (c_int, [c_ptr, c_int, c_i64, c_ptr, c_ptr, c_i64, c_ptr, c_i32, c_i32,
                                            c_i32, c_ptr, c_i64, c_ptr, c_i64, c_ptr, c_ptr, c_i64, c_i32,
                                            c_i32, c_ptr, c_i64, c_ptr, c_size, c_ptr]),
    "idx_paged_mqa_topk_decode_noalloc": (c_int, [c_ptr, c_i64, c_ptr, c_int, c_i64, c_ptr, c_i32,
                                                  c_i32, c_i64, c_ptr, c_i64, c_ptr, c_i32, c_ptr,
                                                  c_i64, c_i32, c_ptr, c_i64, c_ptr]),
    "idx_diag_mma_peak": (c_int, [c_int, c_i32, c_i32, ctypes.POINTER(ctypes.c_double), c_ptr]),
    "idx_diag_l2_read": (c_int, [c_ptr, c_i64, c_i32, c_i32, c_ptr]),
    "idx_block_span": (c_int, [c_i64, c_i64, ctypes.POINTER(c_i32)]),
    "idx_workspace_bytes": (c_size, [c_int, c_i32, c_i32, c_i32]),
    "idx_status_string": (ctypes.c_char_p, [c_int]),
    "idx_last_error": (ctypes.c_char_p, []),
    "idx_device_error": (c_int, [c_ptr]),
}

_LIB = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libidx.so (once). Raises if it has not been built: there is no fallback."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libidx.so not found at {p}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib
