"""The allocation-free decode entry point agrees with the workspace-based entry points.

Some callers of this library cannot allocate device memory (an engine that
plans every buffer ahead of time, a plugin handed only raw pointers), so they
cannot pass the selection workspace. idx_paged_mqa_topk_decode_noalloc keeps
that workspace in a scratch array built into the library. This test calls it
through the C ABI, twice in a row with different queries (the second call
must not see the first call's scratch contents), and compares the scores and
the selections with idx_paged_mqa_logits_decode + idx_topk and with the CPU
oracle. The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_indexer_fp8_gb300 as idx
from oracle import indexer as O
from oracle.codecs import bf16_decode
from sparse_attention_indexer_fp8_gb300 import workloads as W
from tests.checks import assert_logits_close, assert_topk_row, assert_topk_values_exact

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(lib, q, w, cache, block_size, bt, ctx, logits, k, out):
    return lib.idx_paged_mqa_topk_decode_noalloc(
        q.data_ptr(), q.stride(0), w.data_ptr(), 0, w.stride(0), cache.data_ptr(), cache.shape[0],
        block_size, cache.stride(0), bt.data_ptr(), bt.stride(0), ctx.data_ptr(), ctx.shape[0],
        logits.data_ptr(), logits.stride(0), k, out.data_ptr(), out.stride(0),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_workspace_entry_points():
    from sparse_attention_indexer_fp8_gb300.build import build_library

    build_library()
    lib = idx.library()
    ctx = np.array([1000, 2048, 3000, 4096, 5000, 77, 2049, 640, 9000], dtype=np.int32)
    pool = W.make_pool(61, ctx)
    stride = W.block_stride_bytes()
    cache = torch.zeros((pool.num_blocks, stride), dtype=torch.uint8, device=DEV)
    ocache = np.zeros((pool.num_blocks, stride), dtype=np.uint8)
    for b in range(len(ctx)):
        kraw = W.make_k(61, b, int(ctx[b]))
        kb = torch.from_numpy(kraw.view(np.int16)).to(DEV).view(torch.bfloat16)
        idx.idx_k_quant_and_cache(kb, torch.from_numpy(pool.slot_mapping(b)).to(DEV), cache, 64)
        O.k_quant_and_cache(bf16_decode(kraw), pool.slot_mapping(b), ocache, 64)
    bt = torch.from_numpy(pool.block_table).to(DEV)
    dctx = torch.from_numpy(ctx).to(DEV)
    rows = len(ctx)
    ld = (int(ctx.max()) + 63) // 64 * 64
    k = 2048
    for call, seed in enumerate((62, 63)):
        q8, w = W.make_q(seed, rows)
        q, wt = torch.from_numpy(q8).to(DEV), torch.from_numpy(w).to(DEV)
        lg_a = torch.empty((rows, ld), dtype=torch.float32, device=DEV)
        sel_a = torch.empty((rows, k), dtype=torch.int32, device=DEV)
        assert _noalloc(lib, q, wt, cache, 64, bt, dctx, lg_a, k, sel_a) == 0, \
            lib.idx_last_error().decode()
        lg_b = torch.empty((rows, ld), dtype=torch.float32, device=DEV)
        sel_b = torch.empty((rows, k), dtype=torch.int32, device=DEV)
        idx.idx_paged_mqa_logits_decode(q, wt, cache, 64, bt, dctx, lg_b)
        idx.idx_topk(lg_b, None, dctx, k, sel_b)
        idx.idx_device_error()
        a, b_ = lg_a.cpu().numpy(), lg_b.cpu().numpy()
        sa, sb = sel_a.cpu().numpy(), sel_b.cpu().numpy()
        ref = O.paged_decode_logits(q8, w, ocache, 64, pool.block_table, ctx, 1)
        for r in range(rows):
            L = int(ctx[r])
            assert_logits_close(a[r, :L], ref[r, :L], f"call {call} row {r} vs oracle")
            assert_topk_row(sa[r], ref[r, :L], k, f"call {call} row {r} top-k vs oracle")
            assert_logits_close(a[r, :L], b_[r, :L], f"call {call} row {r}")
            assert_topk_values_exact(sa[r], a[r, :L], k, f"call {call} row {r}")
            assert np.array_equal(np.sort(a[r, sa[r][sa[r] >= 0]]), np.sort(b_[r, sb[r][sb[r] >= 0]]))


def test_noalloc_rejects_more_rows_than_its_scratch():
    lib = idx.library()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check fails first
    st = lib.idx_paged_mqa_topk_decode_noalloc(fake, 8192, fake, 0, 64, fake, 8, 64, 8704, fake, 8,
                                               fake, 1025, fake, 4096, 2048, fake, 2048, None)
    assert st == 2 and b"1024" in lib.idx_last_error()
    # a bad k or output stride is refused before anything is enqueued
    for k, ld_out, want in ((0, 2048, 1), (4097, 8192, 2), (2048, 2047, 1)):
        st = lib.idx_paged_mqa_topk_decode_noalloc(fake, 8192, fake, 0, 64, fake, 8, 64, 8704, fake, 8,
                                                   fake, 4, fake, 4096, k, fake, ld_out, None)
        assert st == want, (k, ld_out, st)
