"""The named workloads at full size, in the launch configuration the benchmark times.

Each test runs one whole step through the library (the same entry points,
buffers and selection workspace as bench.py) and checks sampled rows against
the oracle, computed one row at a time: logits within 1e-3 + 2e-3 * |oracle|
(plus bf16 rounding for bf16 scores), top-k sets up to ties within that
tolerance, slots and remaps bit-exact, and the expansion bit-exact on every
row. Large pools draw k with the device generator; the oracle draws the same k
by calling that generator again.
"""

import numpy as np
import pytest
import torch

import sparse_attention_indexer_fp8_gb300 as idx
from oracle import indexer as O
from oracle.codecs import bf16_decode
from sparse_attention_indexer_fp8_gb300 import workloads as W
from sparse_attention_indexer_fp8_gb300.pipeline import (DcpDecodeStep, DecodeStep, HierarchicalStep,
                                                         cache_block_stride, fill_paged_cache)
from tests.checks import assert_logits_close, assert_topk_row

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from sparse_attention_indexer_fp8_gb300.build import build_library

    build_library()
    idx.library()
    yield
    idx.idx_device_error()


def _assert_selection_exact_all_rows(logits, lo, hi, sel, k, what, chunk=512):
    """Every row's selection against the scores the kernel itself wrote (on the GPU, by torch).

    For a row with more than k visible columns [lo, hi): k distinct request-local
    indices whose scores are exactly the k largest visible scores (as a multiset;
    which of several equal scores is kept is free). For a row with at most k
    visible columns: 0..n-1 in order, then -1.
    """
    R = sel.shape[0]
    lo_t = torch.as_tensor(np.asarray(lo, dtype=np.int64), device=DEV)
    hi_t = torch.as_tensor(np.asarray(hi, dtype=np.int64), device=DEV)
    n_t = (hi_t - lo_t).clamp(min=0)
    cols = torch.arange(logits.shape[1], device=DEV)
    ninf = torch.tensor(float("-inf"), device=DEV)
    for r0 in range(0, R, chunk):
        r1 = min(R, r0 + chunk)
        lg = logits[r0:r1].float()
        s = sel[r0:r1].long()
        lo_c, hi_c, n_c = lo_t[r0:r1, None], hi_t[r0:r1, None], n_t[r0:r1]
        big = n_c > k
        if big.any():
            vis = (cols[None, :] >= lo_c) & (cols[None, :] < hi_c)
            want = torch.topk(torch.where(vis, lg, ninf)[big], k, dim=1).values
            idx = s[big]
            assert bool(((idx >= 0) & (idx < n_c[big, None])).all()), f"{what}: index out of range"
            srt = idx.sort(dim=1).values
            assert bool((srt[:, 1:] > srt[:, :-1]).all()), f"{what}: duplicate indices"
            got = torch.gather(lg[big], 1, idx + lo_c[big]).sort(dim=1, descending=True).values
            assert torch.equal(got, want), f"{what}: selected scores differ from the top-{k} scores"
        small = ~big
        if small.any():
            ar = torch.arange(s.shape[1], device=DEV)[None, :]
            expect = torch.where(ar < n_c[small, None], ar, torch.full_like(ar, -1))
            assert torch.equal(s[small][:, :k], expect[:, :k]), f"{what}: short rows must list 0..n-1 then -1"


def _k_host(seed, b, n):
    return bf16_decode(W.make_k_device(seed, b, n, DEV).view(torch.int16).cpu().numpy().view(np.uint16))


def _decode(wl, n_rows, kv="fp8"):
    pool = wl.pool
    cache = torch.zeros((pool.num_blocks, cache_block_stride(kv)), dtype=torch.uint8, device=DEV)
    fill_paged_cache(pool, wl.seed, cache, device_k=True, kv=kv)
    stp = DecodeStep(wl.batch, int(pool.ctx_lens.max()), kv=kv)
    bt = torch.from_numpy(pool.block_table).to(DEV)
    ctx = torch.from_numpy(pool.ctx_lens).to(DEV)
    slots = stp.run(torch.from_numpy(wl.q8).to(DEV), torch.from_numpy(wl.w).to(DEV), cache, bt, ctx)
    idx.idx_device_error()
    _assert_selection_exact_all_rows(stp.logits, np.zeros(wl.batch), pool.ctx_lens, stp.local, wl.topk,
                                     "decode selection")
    lg, loc, sl = stp.logits.cpu().numpy(), stp.local.cpu().numpy(), slots.cpu().numpy()
    assert stp.ws is None or not stp.ws.any().item()
    for b in range(wl.batch):   # the fused slot conversion on every row
        sm = pool.slot_mapping(b)
        L = int(pool.ctx_lens[b])
        assert np.array_equal(sl[b], np.where(loc[b] >= 0, sm[np.clip(loc[b], 0, L - 1)], -1)), f"slots row {b}"
    # the oracle on the longest and the shortest row and a seeded sample of the rest
    rng = np.random.default_rng(wl.seed)
    ends = {int(np.argmax(pool.ctx_lens)), int(np.argmin(pool.ctx_lens))}
    rest = [b for b in range(wl.batch) if b not in ends]
    for b in sorted(ends | set(rng.choice(rest, size=n_rows - len(ends), replace=False).tolist())):
        L = int(pool.ctx_lens[b])
        if kv == "mxfp4":
            ref = O.logits_row_values(wl.q8[b], wl.w[b], O.mxfp4_values(*O.mxfp4_quant(_k_host(wl.seed, b, L))))
        else:
            k8, ks = O.k_quant(_k_host(wl.seed, b, L))
            ref = O.logits_row(wl.q8[b], wl.w[b], k8, ks)
        assert_logits_close(lg[b, :L], ref, f"row {b}")
        assert_topk_row(loc[b], ref, wl.topk, f"top-k row {b}")


def test_long_decode_mxfp4_b128_64k_128k():
    # the long-context decode workload on the MXFP4 indexer cache (the V4.1 format)
    _decode(W.long_decode(), 12, kv="mxfp4")


def test_paged_decode_b64_8k_32k():
    _decode(W.paged_decode(), 12)


def test_long_decode_b128_64k_128k():
    _decode(W.long_decode(), 12)


def test_prefill_chunk_8192_on_32k():
    wl = W.prefill_chunk()
    T, S = wl.q8.shape[0], wl.S
    pool = W.make_pool(wl.seed, [S])
    cache = torch.zeros((pool.num_blocks, W.block_stride_bytes()), dtype=torch.uint8, device=DEV)
    k = W.make_k_device(wl.seed, 0, S, DEV)
    idx.idx_k_quant_and_cache(k, torch.from_numpy(pool.slot_mapping(0)).to(DEV), cache, 64)
    k8 = torch.empty((S, 128), dtype=torch.uint8, device=DEV)
    kscale = torch.empty(S, dtype=torch.float32, device=DEV)
    idx.idx_gather_k(cache, 64, torch.from_numpy(pool.block_table[0]).to(DEV), S, k8, kscale)
    q = torch.from_numpy(wl.q8).to(DEV)
    w = torch.from_numpy(wl.w.view(np.int16)).to(DEV).view(torch.bfloat16)
    ks, ke = torch.from_numpy(wl.row_ks).to(DEV), torch.from_numpy(wl.row_ke).to(DEV)
    logits = torch.empty((T, S), dtype=torch.float32, device=DEV)
    idx.idx_mqa_logits_prefill(q, w, k8, kscale, ks, ke, logits)
    sel = torch.empty((T, wl.topk), dtype=torch.int32, device=DEV)
    idx.idx_topk(logits, ks, ke, wl.topk, sel)
    idx.idx_device_error()
    _assert_selection_exact_all_rows(logits, wl.row_ks, wl.row_ke, sel, wl.topk, "prefill selection")
    ok8, oks = O.k_quant(bf16_decode(k.view(torch.int16).cpu().numpy().view(np.uint16)))
    assert np.array_equal(k8.cpu().numpy(), ok8) and np.array_equal(kscale.cpu().numpy(), oks)
    wv = bf16_decode(wl.w)
    rows = [0, 1, 2, 3, 4, 5, 4095, T - 2, T - 1]
    lg = logits[rows].cpu().numpy()
    sl = sel[rows].cpu().numpy()
    for i, t in enumerate(rows):
        hi = int(wl.row_ke[t])
        ref = O.logits_row(wl.q8[t], wv[t], ok8[:hi], oks[:hi])
        assert_logits_close(lg[i, :hi], ref, f"prefill row {t}")
        assert np.all(np.isneginf(lg[i, hi:])), f"prefill mask row {t}"
        assert_topk_row(sl[i], ref, wl.topk, f"prefill top-k row {t}")


def _hierarchical(wl, check_rows, kv="fp8"):
    pool = wl.pool
    B = len(pool.ctx_lens)
    stride = W.mxfp4_block_stride_bytes() if kv == "mxfp4" else W.block_stride_bytes()
    cache = torch.zeros((pool.num_blocks, stride), dtype=torch.uint8, device=DEV)
    fill_paged_cache(pool, wl.seed, cache, device_k=True, kv=kv)
    stp = HierarchicalStep(B, wl.cand.shape[1], wl.cand_block_size, wl.sbk, wl.topk, kv=kv)
    slots = stp.run(torch.from_numpy(wl.q8).to(DEV), torch.from_numpy(wl.w).to(DEV), cache,
                    torch.from_numpy(pool.block_table).to(DEV), torch.from_numpy(pool.ctx_lens).to(DEV),
                    torch.from_numpy(wl.cand).to(DEV))
    idx.idx_device_error()
    osi, oend = O.expand_candidates(wl.cand, None, pool.ctx_lens, wl.cand_block_size, wl.sbk)
    assert np.array_equal(stp.sparse_idx.cpu().numpy(), osi)
    assert np.array_equal(stp.end.cpu().numpy(), oend)
    assert stp.ws is None or not stp.ws.any().item()
    _assert_selection_exact_all_rows(stp.logits, np.zeros(B), oend, stp.cols, wl.topk, "sparse selection")
    lg = stp.logits.float().cpu().numpy()
    cols, pos, sl = stp.cols.cpu().numpy(), stp.positions.cpu().numpy(), slots.cpu().numpy()
    for b in check_rows:
        e = int(oend[b])
        kall = _k_host(wl.seed, b, int(pool.ctx_lens[b]))
        toks = np.array([O.sparse_column_token(osi[b], c, wl.sbk) for c in range(e)], dtype=np.int64)
        if kv == "mxfp4":
            ref = O.logits_row_values(wl.q8[b], wl.w[b], O.mxfp4_values(*O.mxfp4_quant(kall[toks])))
        else:
            k8, ks = O.k_quant(kall[toks])
            ref = O.logits_row(wl.q8[b], wl.w[b], k8, ks)
        assert_logits_close(lg[b, :e], ref, f"sparse row {b}", bf16=True)
        assert np.all(np.isneginf(lg[b, e:]))
        assert_topk_row(cols[b], ref, wl.topk, f"sparse top-k row {b}", bf16=True)
        m = min(wl.topk, e)
        assert pos[b, :m].tolist() == toks[cols[b, :m]].tolist() and np.all(pos[b, m:] == -1)
        sm = pool.slot_mapping(b)
        assert np.array_equal(sl[b], np.where(pos[b] >= 0, sm[np.clip(pos[b], 0, None)], -1))


def test_hierarchical_b128_128k():
    wl = W.hierarchical()
    rng = np.random.default_rng(wl.seed)
    _hierarchical(wl, sorted(rng.choice(128, size=6, replace=False).tolist()))


def test_hierarchical_mxfp4_b128_128k():
    # the hierarchical workload on the MXFP4 indexer cache (the V4.1 format)
    wl = W.hierarchical()
    rng = np.random.default_rng(wl.seed + 1)
    _hierarchical(wl, sorted(rng.choice(128, size=6, replace=False).tolist()), kv="mxfp4")


def test_hierarchical_many_tiles_per_cta_every_row():
    # 128 rows of 32 sparse tiles each: every CTA walks ~27 tiles across row
    # boundaries, inactive tails and unpaired commit groups; every row is checked
    wl = W.hierarchical(seed=2024, batch=128, ctx=16384, n_cand=64)
    _hierarchical(wl, list(range(0, 128, 1)))


def test_dcp_four_emulated_ranks_paged_decode():
    # Context-parallel decode of the paged decode workload (64 requests of 8K-32K
    # tokens) with four ranks emulated on one GPU: rank r scores the r-th quarter
    # of every request's blocks through its own block table, keeps its local
    # top-2048 with scores, the lists are concatenated rank after rank (the
    # all-gather), and the merge must give the whole context's top-2048.
    wl, world = W.paged_decode(), 4
    pool, B, bs = wl.pool, wl.batch, wl.pool.block_size
    cache = torch.zeros((pool.num_blocks, W.block_stride_bytes()), dtype=torch.uint8, device=DEV)
    fill_paged_cache(pool, wl.seed, cache, device_k=True)
    L = pool.ctx_lens.astype(np.int64)
    nblk = (L + bs - 1) // bs
    starts = np.stack([np.minimum(nblk * r // world * bs, L) for r in range(world + 1)], axis=1)
    q, w = torch.from_numpy(wl.q8).to(DEV), torch.from_numpy(wl.w).to(DEV)
    steps, cv, ci = [], [], []
    for rank in range(world):
        lens = (starts[:, rank + 1] - starts[:, rank]).astype(np.int32)
        bt = np.zeros_like(pool.block_table)
        for b in range(B):
            first, cnt = int(starts[b, rank]) // bs, (int(lens[b]) + bs - 1) // bs
            bt[b, :cnt] = pool.block_table[b, first:first + cnt]
        stp = DcpDecodeStep(B, int(lens.max()), world)
        v, i = stp.select_local(q, w, cache, torch.from_numpy(bt).to(DEV), torch.from_numpy(lens).to(DEV))
        steps.append(stp)
        cv.append(v)
        ci.append(i)
    offs = torch.from_numpy(starts[:, :world].astype(np.int32)).to(DEV)
    pos = steps[0].merge(torch.cat(cv, 1), torch.cat(ci, 1), offs).cpu().numpy()
    sc = steps[0].scores.cpu().numpy()
    idx.idx_device_error()
    assert all(s.ws is None or not s.ws.any().item() for s in steps)
    rng = np.random.default_rng(wl.seed + 1)
    for b in sorted(rng.choice(B, size=4, replace=False).tolist()):
        n = int(L[b])
        k8, ks = O.k_quant(_k_host(wl.seed, b, n))
        ref = O.logits_row(wl.q8[b], wl.w[b], k8, ks)
        assert_topk_row(pos[b], ref, wl.topk, f"dcp top-k row {b}")
        assert_logits_close(sc[b], ref[pos[b]], f"dcp scores row {b}")


def test_q_prep_chunk_8192_bitexact_sampled():
    # the q preparation of the prefill chunk (8192 queries, positions 24576..32767 of
    # a 32K context) in the benchmark's configuration: bf16 q, fp32 weights in,
    # bf16 weights out; q8 bytes and weights bit-exact on 256 sampled rows
    wl = W.q_prep_chunk()
    q = W.make_q_raw_device(wl.seed, wl.T, DEV)
    q8 = torch.empty((wl.T, 8192), dtype=torch.uint8, device=DEV)
    wo = torch.empty((wl.T, 64), dtype=torch.bfloat16, device=DEV)
    idx.idx_q_rope_quant(q, torch.from_numpy(wl.positions).to(DEV), torch.from_numpy(wl.cos_sin).to(DEV),
                         torch.from_numpy(wl.w).to(DEV), q8, wo, 128 ** -0.5, 64 ** -0.5)
    idx.idx_device_error()
    rows = np.sort(np.random.default_rng(wl.seed).choice(wl.T, 256, replace=False))
    rows = np.unique(np.concatenate([rows, [0, wl.T - 1]]))
    qs = bf16_decode(q[rows].view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float32)
    o8, ow, _ = O.q_rope_quant(qs.reshape(-1, 64, 128), wl.positions[rows], wl.cos_sin, wl.w[rows],
                               128 ** -0.5, 64 ** -0.5)
    assert np.array_equal(q8[rows].cpu().numpy().reshape(-1, 64, 128), o8)
    from oracle.codecs import bf16_encode
    assert np.array_equal(wo[rows].view(torch.int16).cpu().numpy().view(np.uint16), bf16_encode(ow))


def test_hierarchical_mtp_b128_128k_four_layers():
    # MTP rows (next_n 2) at 128K with one expansion shared by four layers, as benchmarked
    wl = W.hierarchical_mtp()
    pool, nn = wl.pool, wl.next_n
    B = len(pool.ctx_lens)
    rows = B * nn
    cache = torch.zeros((pool.num_blocks, W.block_stride_bytes()), dtype=torch.uint8, device=DEV)
    fill_paged_cache(pool, wl.seed, cache, device_k=True)
    row_ke = np.array([int(pool.ctx_lens[r // nn]) - nn + r % nn + 1 for r in range(rows)], dtype=np.int32)
    stp = HierarchicalStep(rows, wl.cand.shape[1], wl.cand_block_size, wl.sbk, wl.topk, pool.block_size, DEV,
                           next_n=nn)
    stp.expand(torch.from_numpy(wl.cand).to(DEV), torch.from_numpy(pool.ctx_lens).to(DEV),
               torch.from_numpy(row_ke).to(DEV))
    osi, oend = O.expand_candidates(wl.cand, None, row_ke, wl.cand_block_size, wl.sbk)
    assert np.array_equal(stp.sparse_idx.cpu().numpy(), osi) and np.array_equal(stp.end.cpu().numpy(), oend)
    bt = torch.from_numpy(pool.block_table).to(DEV)
    ctx = torch.from_numpy(pool.ctx_lens).to(DEV)
    rng = np.random.default_rng(wl.seed)
    check = sorted(rng.choice(rows, size=3, replace=False).tolist())
    for layer in range(4):
        q8, w = (wl.q8, wl.w) if layer == 0 else W.make_q(wl.seed + 17 * layer, rows)
        slots = stp.score(torch.from_numpy(q8).to(DEV), torch.from_numpy(w).to(DEV), cache, bt, ctx)
        idx.idx_device_error()
        if layer not in (0, 3):
            continue
        lg = stp.logits.float().cpu().numpy()
        cols, pos, sl = stp.cols.cpu().numpy(), stp.positions.cpu().numpy(), slots.cpu().numpy()
        for r in check:
            e = int(oend[r])
            b = r // nn
            kall = _k_host(wl.seed, b, int(pool.ctx_lens[b]))
            toks = np.array([O.sparse_column_token(osi[r], c, wl.sbk) for c in range(e)], dtype=np.int64)
            k8, ks = O.k_quant(kall[toks])
            ref = O.logits_row(q8[r], w[r], k8, ks)
            assert_logits_close(lg[r, :e], ref, f"layer {layer} mtp row {r}", bf16=True)
            assert_topk_row(cols[r], ref, wl.topk, f"layer {layer} mtp top-k row {r}", bf16=True)
            m = min(wl.topk, e)
            assert pos[r, :m].tolist() == toks[cols[r, :m]].tolist() and np.all(pos[r, m:] == -1)
            sm = pool.slot_mapping(b)
            assert np.array_equal(sl[r], np.where(pos[r] >= 0, sm[np.clip(pos[r], 0, None)], -1))
    assert stp.ws is None or not stp.ws.any().item()
