"""The C-ABI library loads and exports every entry point of include/idx.h (CPU only).

Also exercises the host-only entry points and argument validation paths that
return before any CUDA call.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_fp8_gb300 import _lib
    from sparse_attention_indexer_fp8_gb300.build import build_library

    build_library()
    return _lib.load()


def _declared():
    with open(os.path.join(ROOT, "include", "idx.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\S.*?\b(idx_\w+)\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared()
    for required in ("idx_k_quant_and_cache", "idx_mqa_logits_prefill", "idx_paged_mqa_logits_decode",
                     "idx_topk", "idx_expand_candidates", "idx_sparse_topk_remap",
                     "idx_req_to_global_slots"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from sparse_attention_indexer_fp8_gb300 import _lib

    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding has no signature for {name}"


def test_host_helpers(lib):
    span = ctypes.c_int32(0)
    assert lib.idx_block_span(8704, 128, ctypes.byref(span)) == 0 and span.value == 68
    assert lib.idx_block_span(8704, 132, ctypes.byref(span)) == 2   # not divisible -> unsupported
    assert b"does not" not in lib.idx_status_string(0)
    assert lib.idx_status_string(2) == b"unsupported configuration"
    assert b"multiple" in lib.idx_last_error()
    assert lib.idx_block_span(0, 128, ctypes.byref(span)) == 1
    assert lib.idx_workspace_bytes(5, 128, 131072, 2048) == 128 * 1024 * 4
    assert lib.idx_workspace_bytes(1, 128, 131072, 2048) == 0
    # max_cols 0: the buffer's size whatever the rows' length
    assert lib.idx_workspace_bytes(7, 8192, 0, 2048) == 8192 * 1024 * 4
    # many rows of at most 4096 columns need none on a device with fewer SMs than
    # rows; without a device the full size is returned
    assert lib.idx_workspace_bytes(7, 8192, 4096, 2048) in (0, 8192 * 1024 * 4)
    assert lib.idx_workspace_bytes(7, 0, 4096, 2048) == 0


def test_validation_rejects_before_touching_the_device(lib):
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: every call below fails validation first
    # block size outside {16, 32, 64, 128}
    assert lib.idx_k_quant_and_cache(fake, 1, 128, 4, fake, fake, 8, 48, 8704, 0, None) == 2
    assert lib.idx_k_quant_and_cache(fake, 1, 128, 4, fake, fake, 8, 64, 8704, 2, None) == 2   # scale_fmt
    # block stride too small for 64 tokens of 132 bytes
    assert lib.idx_k_quant_and_cache(fake, 1, 128, 4, fake, fake, 8, 64, 8000, 0, None) == 1
    # k above the selection limit, NULL logits
    assert lib.idx_topk(fake, 0, 4096, None, fake, 4, 5000, fake, 5000, None, 0, None, 0, None) == 2
    assert lib.idx_topk(None, 0, 4096, None, fake, 4, 2048, fake, 2048, None, 0, None, 0, None) == 1
    # q preparation: bad rope style, short stride, bad dtype
    assert lib.idx_q_rope_quant(fake, 1, 8192, fake, fake, 64, 10, 5, fake, 0, 64, 1.0, 1.0, 4, fake,
                                8192, fake, 0, 64, None) == 2
    assert lib.idx_q_rope_quant(fake, 1, 100, fake, fake, 64, 10, 0, fake, 0, 64, 1.0, 1.0, 4, fake,
                                8192, fake, 0, 64, None) == 1
    assert lib.idx_q_rope_quant(fake, 7, 8192, fake, fake, 64, 10, 0, fake, 0, 64, 1.0, 1.0, 4, fake,
                                8192, fake, 0, 64, None) == 2
    # merge: candidate stride smaller than n_shards * k_local
    assert lib.idx_dcp_topk_merge(fake, 100, fake, 100, fake, 0, 4, 1, 2048, 2, 2048, fake, 2048, None,
                                  0, None) == 1
    # per-row offsets narrower than the shard count; position stride 0
    assert lib.idx_dcp_topk_merge(fake, 8192, fake, 8192, fake, 2, 4, 1, 2048, 2, 2048, fake, 2048, None,
                                  0, None) == 1
    assert lib.idx_dcp_topk_merge(fake, 8192, fake, 8192, fake, 0, 4, 0, 2048, 2, 2048, fake, 2048, None,
                                  0, None) == 1
    assert lib.idx_dcp_topk_merge(fake, 8192, fake, 8192, fake, 0, 4, 1, 2048, 2, 5000, fake, 5000, None,
                                  0, None) == 2
    # candidate count not a power of two
    assert lib.idx_expand_candidates(fake, 64, 4, 48, None, fake, 64, 64, fake, 64, fake, None) == 2
    # block_span smaller than block_size
    assert lib.idx_req_to_global_slots(fake, 8, 1, 8, None, fake, 8, 64, 32, fake, 8, None) == 2
    # fused slot conversion: the same checks (span, NULL slots, slot stride)
    assert lib.idx_topk_slots(fake, 0, 4096, None, fake, 4, 2048, fake, 2048, None, fake, 8, 64, 32,
                              fake, 2048, None, 0, None) == 2
    assert lib.idx_topk_slots(fake, 0, 4096, None, fake, 4, 2048, fake, 2048, None, fake, 8, 64, 64,
                              None, 2048, None, 0, None) == 1
    assert lib.idx_sparse_topk_remap_slots(fake, 1, 4096, fake, fake, 64, None, 64, 4, 2048, None, 0,
                                           fake, 2048, None, fake, 8, 64, 64, fake, 100, None, 0,
                                           None) == 1
    # dense decode with next_n = 3
    assert lib.idx_paged_mqa_logits_decode(fake, 8192, fake, 0, 64, fake, 16, 64, 8704, fake, 8, fake,
                                           2, 3, None, 0, 0, None, 0, fake, 0, 4096, None, 0, None) == 2
    # MXFP4 cache: stride below 64 * 68, stride not a multiple of 32, block size, misaligned cache
    assert lib.idx_k_quant_and_cache_mxfp4(fake, 1, 128, 4, fake, fake, 8, 64, 4350, None) == 1
    assert lib.idx_k_quant_and_cache_mxfp4(fake, 1, 128, 4, fake, fake, 8, 64, 4368, None) == 2
    assert lib.idx_k_quant_and_cache_mxfp4(fake, 1, 128, 4, fake, fake, 8, 48, 4608, None) == 2
    assert lib.idx_k_quant_and_cache_mxfp4(fake, 1, 128, 4, fake, ctypes.c_void_p(0x1010), 8, 64, 4608,
                                           None) == 2
    # MXFP4 decode: dense next_n 2, a stride that is not a multiple of 32, too small a stride
    assert lib.idx_paged_mqa_logits_decode_mxfp4(fake, 8192, fake, 0, 64, fake, 16, 64, 4608, fake, 8, fake,
                                                 2, 2, None, 0, 0, None, 0, fake, 0, 4096, None, 0, None) == 2
    assert lib.idx_paged_mqa_logits_decode_mxfp4(fake, 8192, fake, 0, 64, fake, 16, 64, 4368, fake, 8, fake,
                                                 2, 1, None, 0, 0, None, 0, fake, 0, 4096, None, 0, None) == 2
    assert lib.idx_paged_mqa_logits_decode_mxfp4(fake, 8192, fake, 0, 64, fake, 16, 64, 4096, fake, 8, fake,
                                                 2, 1, None, 0, 0, None, 0, fake, 0, 4096, None, 0, None) == 1
    # MXFP4 prefill gather: block size, stride, NULL output
    assert lib.idx_gather_k_mxfp4(fake, 48, 4608, fake, 10, fake, fake, None) == 2
    assert lib.idx_gather_k_mxfp4(fake, 64, 4368, fake, 10, fake, fake, None) == 2
    assert lib.idx_gather_k_mxfp4(fake, 64, 4608, fake, 10, None, fake, None) == 1
    # MXFP4 prefill scoring: the dense mode does not exist, codes must be 32-byte aligned
    assert lib.idx_mqa_logits_prefill_mxfp4(fake, 8192, fake, 0, 64, fake, fake, 64, None, None, 4, None, 0,
                                            0, None, 0, fake, 0, 64, None, 0, None) == 2
    assert lib.idx_mqa_logits_prefill_mxfp4(fake, 8192, fake, 0, 64, ctypes.c_void_p(0x1010), fake, 64, None,
                                            None, 4, fake, 1, 1, fake, 64, fake, 1, 64, None, 0, None) == 2
    # tensor-rate diagnostic: unknown kind, no iterations
    assert lib.idx_diag_mma_peak(7, 100, 0, None, None) == 2
    assert lib.idx_diag_mma_peak(0, 0, 0, None, None) == 1
    assert lib.idx_diag_l2_read(None, 1 << 20, 1, 0, None) == 1              # NULL buffer
    assert lib.idx_diag_l2_read(fake, 15, 1, 0, None) == 1                   # not a multiple of 16
    assert lib.idx_diag_l2_read(ctypes.c_void_p(0x1008), 1 << 20, 1, 0, None) == 1   # unaligned
    assert lib.idx_diag_l2_read(fake, 1 << 20, 0, 0, None) == 1              # passes < 1
    # misaligned q stride
    assert lib.idx_mqa_logits_prefill(fake, 8200, fake, 0, 64, fake, fake, 64, None, fake, 4, None, 0,
                                      0, None, 0, fake, 0, 64, None, 0, None) == 2
