"""Parity of every CUDA entry point with the CPU oracle on small seeded inputs.

Sizes span several 128-token tiles, ragged tails, every supported block size,
strided inputs and outputs, and the degenerate cases (empty rows, rows with at
most k visible tokens, all-equal scores). Integer and byte outputs must match
bit for bit; logits within 1e-3 + 2e-3 * |oracle|; top-k sets exactly up to
ties within that tolerance.
"""

import numpy as np
import pytest
import torch

import sparse_attention_indexer_fp8_gb300 as idx
from oracle import indexer as O
from oracle.codecs import bf16_decode, bf16_encode, e4m3_decode
from sparse_attention_indexer_fp8_gb300 import workloads as W
from tests.checks import assert_logits_close, assert_topk_row, assert_topk_values_exact

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from sparse_attention_indexer_fp8_gb300.build import build_library

    build_library()
    idx.library()
    yield
    idx.idx_device_error()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def dev_bf16(u16):
    return dev(np.asarray(u16, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def host_bf16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def build_caches(pool, seed, block_size=64, stride=None, ue8m0=False):
    """GPU cache filled by the kernel, oracle cache filled by the oracle, same k."""
    stride = stride or W.block_stride_bytes(block_size)
    gcache = torch.zeros((pool.num_blocks, stride), dtype=torch.uint8, device=DEV)
    ocache = np.zeros((pool.num_blocks, stride), dtype=np.uint8)
    ks = []
    for b in range(len(pool.ctx_lens)):
        kb = W.make_k(seed, b, int(pool.ctx_lens[b]))
        ks.append(kb)
        O.k_quant_and_cache(bf16_decode(kb), pool.slot_mapping(b), ocache, block_size, ue8m0)
    k_all = dev_bf16(np.concatenate(ks))
    slots = dev(np.concatenate([pool.slot_mapping(b) for b in range(len(pool.ctx_lens))]))
    idx.idx_k_quant_and_cache(k_all, slots, gcache, block_size, ue8m0=ue8m0)
    return gcache, ocache


# ------------------------------------------------------------------ a1 k quant + insert

def test_k_quant_and_cache_bitexact_tiny_pool():
    wl = W.tiny_decode()
    g, o = build_caches(wl.pool, wl.seed)
    assert np.array_equal(g.cpu().numpy(), o)


def test_ue8m0_cache_bitexact_and_decode_logits():
    # power-of-two k scales (the UE8M0 scale format): the cache bytes equal the
    # oracle's, and the scoring kernels read that cache unchanged
    wl = W.tiny_decode()
    pool = wl.pool
    g, o = build_caches(pool, wl.seed, ue8m0=True)
    assert np.array_equal(g.cpu().numpy(), o)
    rows = len(pool.ctx_lens)
    ld = int(pool.ctx_lens.max())
    out = torch.empty((rows, ld), dtype=torch.float32, device=DEV)
    idx.idx_paged_mqa_logits_decode(dev(wl.q8), dev(wl.w), g, 64, dev(pool.block_table), dev(pool.ctx_lens), out)
    ref = O.paged_decode_logits(wl.q8, wl.w, o, 64, pool.block_table, pool.ctx_lens)
    got = out.cpu().numpy()
    for r in range(rows):
        L = int(pool.ctx_lens[r])
        assert_logits_close(got[r, :L], ref[r, :L], f"ue8m0 row {r}")


def test_k_quant_skips_negative_and_out_of_range_slots_f32_strided_bs16():
    rng = np.random.default_rng(4)
    bs, nb = 16, 40
    stride = W.block_stride_bytes(bs)
    n = 300
    k = (rng.standard_normal((n, 192)) * rng.uniform(0.01, 50, (n, 1))).astype(np.float32)
    slots = rng.permutation(nb * bs)[:n].astype(np.int64)
    slots[::17] = -1
    slots[5] = nb * bs + 3                      # beyond the pool: skipped
    gk = dev(k)[:, :128]                         # ld_k = 192
    gcache = torch.zeros((nb, stride), dtype=torch.uint8, device=DEV)
    idx.idx_k_quant_and_cache(gk, dev(slots), gcache, bs)
    ocache = np.zeros((nb, stride), dtype=np.uint8)
    keep = slots < nb * bs
    O.k_quant_and_cache(k[keep, :128], slots[keep], ocache, bs)
    assert np.array_equal(gcache.cpu().numpy(), ocache)


def test_k_quant_special_values():
    k = np.zeros((6, 128), dtype=np.float32)
    k[1, 3] = 448.0
    k[2, :] = np.float32(1e-45)                  # amax / 448 underflows: scale 0
    k[3, :] = np.linspace(-1e30, 1e30, 128, dtype=np.float32)
    k[4, :] = -0.0
    k[5, :] = np.float32(2.0) ** np.arange(-64, 64, dtype=np.float32)
    bs = 32
    stride = W.block_stride_bytes(bs)
    slots = np.array([0, 5, 33, 40, 63, 64], dtype=np.int64)
    gcache = torch.zeros((3, stride), dtype=torch.uint8, device=DEV)
    idx.idx_k_quant_and_cache(dev(k), dev(slots), gcache, bs)
    ocache = np.zeros((3, stride), dtype=np.uint8)
    O.k_quant_and_cache(k, slots, ocache, bs)
    assert np.array_equal(gcache.cpu().numpy(), ocache)


def test_gather_k_matches_oracle():
    wl = W.tiny_decode()
    g, o = build_caches(wl.pool, wl.seed)
    b = 2
    L = int(wl.pool.ctx_lens[b])
    k8 = torch.empty((L, 128), dtype=torch.uint8, device=DEV)
    ks = torch.empty(L, dtype=torch.float32, device=DEV)
    idx.idx_gather_k(g, 64, dev(wl.pool.block_table[b]), L, k8, ks)
    ok8, oks = O.gather_k(o, 64, wl.pool.block_table[b], L)
    assert np.array_equal(k8.cpu().numpy(), ok8) and np.array_equal(ks.cpu().numpy(), oks)


# ------------------------------------------------------------------ a4 decode logits

@pytest.mark.parametrize("next_n,block_size,out_bf16,w_bf16", [
    (1, 64, False, False), (2, 64, True, False), (4, 64, False, True), (1, 16, False, False),
    (1, 32, True, True), (2, 128, False, False)])
def test_decode_dense_logits(next_n, block_size, out_bf16, w_bf16):
    ctx = np.array([1000, 2048, 3000, 4096, 1, 5, 130, 127], dtype=np.int32)
    ctx = np.maximum(ctx, next_n)
    pool = W.make_pool(77 + next_n, ctx, block_size=block_size, extra_blocks=7)
    g, o = build_caches(pool, 77, block_size)
    rows = len(ctx) * next_n
    q8, w = W.make_q(78, rows, w_bf16=w_bf16)
    # strided q and w: slices of larger buffers
    qbig = np.zeros((rows, 2, 64, 128), dtype=np.uint8)
    qbig[:, 0] = q8
    gq = dev(qbig.reshape(rows, 2 * 64, 128))[:, :64, :]
    wbig = np.zeros((rows, 80), dtype=w.dtype)
    wbig[:, :64] = w
    gw = (dev_bf16(wbig) if w_bf16 else dev(wbig))[:, :64]
    L_max = int(ctx.max())
    out = torch.full((rows, L_max + 40), 7.0, device=DEV,
                     dtype=torch.bfloat16 if out_bf16 else torch.float32)
    idx.idx_paged_mqa_logits_decode(gq, gw, g, block_size, dev(pool.block_table), dev(ctx), out,
                                    next_n=next_n)
    wv = bf16_decode(w) if w_bf16 else w
    ref = O.paged_decode_logits(q8, wv, o, block_size, pool.block_table, ctx, next_n)
    got = out.float().cpu().numpy()
    for r in range(rows):
        L = int(ctx[r // next_n])
        assert_logits_close(got[r, :L], ref[r, :L], f"row {r}", bf16=out_bf16)
        assert np.all(got[r, L:] == 7.0), "columns beyond the context must stay untouched"


def _hier_inputs(seed, block_size=64):
    ctx = np.array([1000, 777, 4096, 2500, 64, 3], dtype=np.int32)
    pool = W.make_pool(seed, ctx, block_size=block_size)
    g, o = build_caches(pool, seed, block_size)
    q8, w = W.make_q(seed, len(ctx))
    cand = W.make_candidates(seed, len(ctx), 16, 64, n_dup=3, n_pad=2, n_oob=2)
    return ctx, pool, g, o, q8, w, cand


def _slots_closed_form(v, bt, req, block_size, block_span):
    """Slot of request-local position v of a row of request req (-1 passes through)."""
    if v < 0 or v // block_size >= bt.shape[1]:
        return -1
    return int(bt[req, v // block_size]) * block_span + v % block_size


@pytest.mark.parametrize("with_ws", [False, True])
def test_topk_with_fused_slots(with_ws):
    # the fused conversion writes, for the same selection, exactly the slots of the
    # closed form (a wider block span and an explicit, permuted row -> request map)
    ctx, pool, g, o, q8, w, cand = _hier_inputs(83)
    rows, k, span = len(ctx), 2048, 96
    L = int(ctx.max())
    logits = torch.empty((rows, (L + 63) // 64 * 64), dtype=torch.float32, device=DEV)
    ws = torch.zeros((rows, 1024), dtype=torch.int32, device=DEV) if with_ws else None
    bt = dev(pool.block_table)
    idx.idx_paged_mqa_logits_decode(dev(q8), dev(w), g, 64, bt, dev(ctx), logits, ws=ws)
    sel = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    slots = torch.full((rows, k + 2), -7, dtype=torch.int32, device=DEV)
    r2q = np.arange(rows, dtype=np.int32)[::-1].copy()
    # rows see the columns of their own request; the slots go through the mapped request's table
    idx.idx_topk(logits, None, dev(ctx), k, sel, ws=ws, slots=slots[:, :k], block_table=bt, block_size=64,
                 block_span=span, row_to_req=dev(r2q))
    idx.idx_device_error()
    sel, sl = sel.cpu().numpy(), slots.cpu().numpy()
    lg = logits.cpu().numpy()
    for r in range(rows):
        assert_topk_values_exact(sel[r], lg[r, :ctx[r]], k, f"row {r}")
        want = [_slots_closed_form(int(v), pool.block_table, int(r2q[r]), 64, span) for v in sel[r]]
        assert sl[r, :k].tolist() == want, r
        assert np.all(sl[r, k:] == -7)


def test_sparse_remap_with_fused_slots():
    ctx, pool, g, o, q8, w, cand = _hier_inputs(84)
    rows, k, sbk = len(ctx), 256, 64
    si = torch.empty((rows, 16), dtype=torch.int32, device=DEV)
    end = torch.empty(rows, dtype=torch.int32, device=DEV)
    idx.idx_expand_candidates(dev(cand), None, dev(ctx), 64, sbk, si, end)
    bt = dev(pool.block_table)
    out = torch.empty((rows, 16 * sbk), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros((rows, 1024), dtype=torch.int32, device=DEV)
    idx.idx_paged_mqa_logits_decode(dev(q8), dev(w), g, 64, bt, dev(ctx), out, sparse_idx=si, end=end,
                                    sbk=sbk, ws=ws)
    pos = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    cols = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    slots = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    idx.idx_sparse_topk_remap(out, end, si, None, sbk, k, pos, col_scratch=cols, ws=ws, slots=slots,
                              block_table=bt, block_size=64, block_span=64)
    # the two-call sequence on the same positions gives the same slots
    ref = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    idx.idx_req_to_global_slots(pos, None, bt, 64, 64, ref)
    idx.idx_device_error()
    assert torch.equal(slots, ref)
    pos, cols, sih = pos.cpu().numpy(), cols.cpu().numpy(), si.cpu().numpy()
    e = end.cpu().numpy()
    lg = out.float().cpu().numpy()
    for r in range(rows):
        m = min(k, int(e[r]))
        assert_topk_values_exact(cols[r], lg[r, :e[r]], k, f"row {r}")
        assert [O.sparse_column_token(sih[r], int(c), sbk) for c in cols[r, :m]] == pos[r, :m].tolist()


@pytest.mark.parametrize("sbk,cbs,out_bf16", [(64, 64, True), (16, 64, True), (8, 16, False),
                                              (32, 64, False)])
def test_decode_sparse_logits_and_remap(sbk, cbs, out_bf16):
    ctx, pool, g, o, q8, w, cand = _hier_inputs(90 + sbk)
    rows = len(ctx)
    R = cbs // sbk
    si = torch.empty((rows, cand.shape[1] * R), dtype=torch.int32, device=DEV)
    end = torch.empty(rows, dtype=torch.int32, device=DEV)
    idx.idx_expand_candidates(dev(cand), None, dev(ctx), cbs, sbk, si, end)
    osi, oend = O.expand_candidates(cand, None, ctx, cbs, sbk)
    assert np.array_equal(si.cpu().numpy(), osi) and np.array_equal(end.cpu().numpy(), oend)
    ncols = si.shape[1] * sbk
    out = torch.empty((rows, ncols), device=DEV, dtype=torch.bfloat16 if out_bf16 else torch.float32)
    idx.idx_paged_mqa_logits_decode(dev(q8), dev(w), g, 64, dev(pool.block_table), dev(ctx), out,
                                    sparse_idx=si, end=end, sbk=sbk)
    ref = O.sparse_logits_decode(q8, w, o, 64, pool.block_table, None, osi, oend, sbk)
    got = out.float().cpu().numpy()
    assert_logits_close(got, ref, "sparse logits", bf16=out_bf16)
    # selection + remap on the kernel's own sparse scores
    k = 300
    pos = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    cols = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    idx.idx_sparse_topk_remap(out, end, si, None, sbk, k, pos, col_scratch=cols)
    pos, cols = pos.cpu().numpy(), cols.cpu().numpy()
    for r in range(rows):
        e = int(oend[r])
        assert_topk_values_exact(cols[r], got[r, :e], k, f"sparse top-k row {r}")
        m = min(k, e)
        for c, p_ in zip(cols[r, :m], pos[r, :m]):
            assert O.sparse_column_token(osi[r], int(c), sbk) == p_
        assert np.all(pos[r, m:] == -1)
        assert_topk_row(cols[r], ref[r, :e], k, f"sparse top-k vs oracle row {r}",
                        bf16=out_bf16)


@pytest.mark.parametrize("next_n", [2, 3])
def test_hierarchical_mtp_rows_and_layer_reuse(next_n):
    # V4.1 consumer layers with multi-token prediction: each request has next_n
    # query rows (row r of request r // next_n sees [0, L - next_n + j + 1)); the
    # expansion is done once and two layers (different q / weights) are scored
    # on it, each checked against the oracle, and the expansion is untouched.
    from sparse_attention_indexer_fp8_gb300.pipeline import HierarchicalStep

    ctx = np.array([1000, 777, 4096, 2500, 64, 5], dtype=np.int32)
    B = len(ctx)
    rows = B * next_n
    pool = W.make_pool(300 + next_n, ctx)
    g, o = build_caches(pool, 300 + next_n)
    cand = W.make_candidates(310 + next_n, rows, 16, 64, n_dup=3, n_pad=2, n_oob=2)
    r2r = np.repeat(np.arange(B), next_n).astype(np.int32)
    row_ke = np.array([O.decode_row_limit(int(ctx[r // next_n]), next_n, r % next_n) for r in range(rows)],
                      dtype=np.int32)
    k = 200
    st = HierarchicalStep(rows, cand.shape[1], 64, 64, k, 64, DEV, next_n=next_n)
    st.expand(dev(cand), dev(ctx), dev(row_ke))
    osi, oend = O.expand_candidates(cand, None, row_ke, 64, 64)
    si0, end0 = st.sparse_idx.clone(), st.end.clone()
    assert np.array_equal(si0.cpu().numpy(), osi) and np.array_equal(end0.cpu().numpy(), oend)
    for layer in range(2):
        q8, w = W.make_q(320 + 10 * layer + next_n, rows)
        slots = st.score(dev(q8), dev(w), g, dev(pool.block_table), dev(ctx)).cpu().numpy()
        assert torch.equal(st.sparse_idx, si0) and torch.equal(st.end, end0), "expansion must be reusable"
        ref = O.sparse_logits_decode(q8, w, o, 64, pool.block_table, r2r, osi, oend, 64)
        got = st.logits.float().cpu().numpy()
        assert_logits_close(got, ref, f"layer {layer} sparse logits", bf16=True)
        cols, pos = st.cols.cpu().numpy(), st.positions.cpu().numpy()
        for r in range(rows):
            e = int(oend[r])
            assert_topk_values_exact(cols[r], got[r, :e], k, f"layer {layer} row {r}")
            assert_topk_row(cols[r], ref[r, :e], k, f"layer {layer} row {r} vs oracle", bf16=True)
            m = min(k, e)
            want = [O.sparse_column_token(osi[r], int(c), 64) for c in cols[r, :m]]
            assert pos[r, :m].tolist() == want and np.all(pos[r, m:] == -1)
        oslots = O.req_to_global_slots(pos, r2r, pool.block_table, 64, 64)
        assert np.array_equal(slots, oslots)


# ------------------------------------------------------------------ a3 prefill logits

@pytest.mark.parametrize("T,w_bf16,out_bf16,ragged", [(256, False, False, False), (255, True, True, True),
                                                      (7, False, False, True)])
def test_prefill_dense_logits(T, w_bf16, out_bf16, ragged):
    S = 4096 if T > 7 else 300
    k8, kscale = W.make_random_cache_tokens(31, S)
    q8, w = W.make_q(32, T, w_bf16=w_bf16)
    if ragged:
        rng = np.random.default_rng(5)
        ks = rng.integers(0, S, T).astype(np.int32)
        ke = np.minimum(ks + rng.integers(0, S, T), S).astype(np.int32)
        ke[::9] = ks[::9]                           # empty rows
    else:
        ks = np.zeros(T, dtype=np.int32)
        ke = np.arange(S - T, S, dtype=np.int32) + 1
    out = torch.empty((T, S + 8), device=DEV, dtype=torch.bfloat16 if out_bf16 else torch.float32)
    idx.idx_mqa_logits_prefill(dev(q8), dev_bf16(w) if w_bf16 else dev(w), dev(k8), dev(kscale),
                               dev(ks), dev(ke), out)
    wv = bf16_decode(w) if w_bf16 else w
    ref = O.mqa_logits(q8, wv, k8, kscale, ks, ke)
    assert_logits_close(out.float().cpu().numpy()[:, :S], ref, "prefill logits",
                        bf16=out_bf16)


def test_prefill_sparse_logits():
    S, T, sbk = 3000, 40, 16
    k8, kscale = W.make_random_cache_tokens(41, S)
    q8, w = W.make_q(42, T)
    rng = np.random.default_rng(6)
    ks = (rng.integers(0, 60, T) * sbk).astype(np.int32)
    ke = np.minimum(ks + rng.integers(1, 2000, T), S).astype(np.int32)
    cand = W.make_candidates(43, T, 16, 40)
    si = torch.empty((T, 64), dtype=torch.int32, device=DEV)
    end = torch.empty(T, dtype=torch.int32, device=DEV)
    idx.idx_expand_candidates(dev(cand), dev(ks), dev(ke), 64, sbk, si, end)
    osi, oend = O.expand_candidates(cand, ks, ke, 64, sbk)
    assert np.array_equal(si.cpu().numpy(), osi) and np.array_equal(end.cpu().numpy(), oend)
    out = torch.empty((T, 64 * sbk), device=DEV, dtype=torch.float32)
    idx.idx_mqa_logits_prefill(dev(q8), dev(w), dev(k8), dev(kscale), dev(ks), dev(ke), out,
                               sparse_idx=si, end=end, sbk=sbk)
    ref = O.sparse_logits_prefill(q8, w, k8, kscale, osi, oend, sbk)
    assert_logits_close(out.cpu().numpy(), ref, "sparse prefill logits")
    k = 512
    pos = torch.empty((T, k), dtype=torch.int32, device=DEV)
    cols = torch.empty((T, k), dtype=torch.int32, device=DEV)
    idx.idx_sparse_topk_remap(out, end, si, dev(ks), sbk, k, pos, col_scratch=cols)
    pos, cols = pos.cpu().numpy(), cols.cpu().numpy()
    for r in range(T):
        e = int(oend[r])
        # the chosen sparse columns against the oracle's sparse scores (tie-tolerant) ...
        assert_topk_row(cols[r], ref[r, :e], k, f"sparse prefill top-k row {r}")
        # ... and each position is the oracle's remap of its column (ks > 0 rows included)
        m = min(k, e)
        expect = O.sparse_remap_columns(cols[r, :m], osi[r], int(ks[r]), sbk)
        assert np.array_equal(pos[r, :m], expect) and np.all(pos[r, m:] == -1)
        assert np.all(pos[r, :m] == np.array([O.sparse_column_token(osi[r], int(c), sbk) for c in cols[r, :m]],
                                             dtype=np.int64) - int(ks[r]))


# ------------------------------------------------------------------ a5 top-k

def _run_topk(x, ks, ke, k, bf16=False, ld_pad=0, out_pad=0):
    rows, width = x.shape
    if bf16:
        xb = bf16_encode(x)
        buf = np.zeros((rows, width + ld_pad), dtype=np.uint16)
        buf[:, :width] = xb
        t = dev_bf16(buf)
        vals = bf16_decode(xb)
    else:
        buf = np.zeros((rows, width + ld_pad), dtype=np.float32)
        buf[:, :width] = x
        t = dev(buf)
        vals = x
    out = torch.full((rows, k + out_pad), -7, dtype=torch.int32, device=DEV)
    idx.idx_topk(t, None if ks is None else dev(ks), dev(ke), k, out)
    return out.cpu().numpy(), vals


@pytest.mark.parametrize("width,k", [(100, 2048), (2048, 2048), (2049, 2048), (5000, 2048),
                                     (40000, 2048), (5000, 1), (5000, 4096), (3000, 777)])
def test_topk_random(width, k):
    x = W.make_logits(width + k, 6, width)
    rng = np.random.default_rng(width)
    ks = rng.integers(0, max(width // 3, 1), 6).astype(np.int32)
    ke = np.minimum(ks + rng.integers(width // 2, width + 1, 6), width).astype(np.int32)
    ke[0], ks[0] = width, 0
    out, vals = _run_topk(x, ks, ke, k, ld_pad=5, out_pad=3)
    for r in range(6):
        seg = vals[r, ks[r]:ke[r]]
        assert_topk_values_exact(out[r], seg, k, f"row {r}")
        assert np.all(out[r, k:] == -7), "columns beyond k must stay untouched"
        ref = O.topk_row(vals[r], ks[r], ke[r], k)
        if len(np.unique(seg)) == len(seg):      # no ties: the index set is unique
            assert set(out[r, :k].tolist()) == set(ref.tolist())


@pytest.mark.parametrize("bf16,width,k,with_ws", [(False, 4096, 2048, False), (True, 4096, 2048, True),
                                                   (False, 1000, 300, True), (True, 3000, 4096, False)])
def test_topk_many_short_rows(bf16, width, k, with_ws):
    # more rows than SMs of at most 4096 columns take the shared-memory selection:
    # ragged ranges with ks > 0, rows with no more visible columns than k, ties
    # and special values; the scores, optional values and the workspace path
    rows = 400
    rng = np.random.default_rng(width + k + bf16)
    x = W.make_logits(width + 11, rows, width, ties=True)
    x[1, :] = 0.5                                        # all equal
    x[2, ::5] = -np.inf
    x[3, 7], x[3, 8], x[3, 9] = np.inf, -np.inf, np.float32(-0.0)
    ks = (rng.integers(0, width // 4, rows)).astype(np.int32)
    ke = np.minimum(ks + rng.integers(1, width + 1, rows), width).astype(np.int32)
    ks[:4], ke[:4] = 0, width
    ke[5] = ks[5] + min(k, width - ks[5])                # exactly k visible (or all of a short row)
    ke[6] = ks[6] + 1
    if bf16:
        xb = bf16_encode(x)
        t = dev_bf16(xb)
        vals = bf16_decode(xb)
    else:
        t = dev(x)
        vals = x
    ws = None
    if with_ws:
        # the first-digit histogram the scoring kernel would have accumulated
        keys = _keys(vals.astype(np.float32).view(np.uint32))
        h = np.zeros((rows, 1024), dtype=np.int32)
        for r in range(rows):
            np.add.at(h[r], (keys[r, ks[r]:ke[r]] >> 22).astype(np.int64), 1)
        ws = dev(h)
    out = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    v = torch.empty((rows, k), dtype=torch.float32, device=DEV)
    idx.idx_topk(t, dev(ks), dev(ke), k, out, vals=v, ws=ws)
    idx.idx_device_error()
    if ws is not None:
        assert not ws.any().item(), "the selection hands the workspace back zeroed"
    out, v = out.cpu().numpy(), v.cpu().numpy()
    for r in range(rows):
        seg = vals[r, ks[r]:ke[r]]
        assert_topk_values_exact(out[r], seg, k, f"row {r}")
        n = int(ke[r] - ks[r])
        got = out[r][out[r] >= 0]
        assert len(got) == min(k, n) and len(set(got.tolist())) == len(got)
        assert np.all(out[r, min(k, n):] == -1)
        if n <= k:
            assert out[r, :n].tolist() == list(range(n)), f"row {r}: all visible columns in order"
        sel = out[r, :min(k, n)]
        assert np.array_equal(v[r, :min(k, n)].view(np.uint32), seg[sel].astype(np.float32).view(np.uint32))
        assert np.all(np.isneginf(v[r, min(k, n):]))


def test_sparse_remap_many_short_rows_with_slots():
    # 300 sparse rows (more than SMs): the shared-memory selection with the remap
    # (ks > 0), the fused slot conversion and the column scratch
    rows, sbk, k = 300, 32, 256
    rng = np.random.default_rng(91)
    n_si = 16
    si = np.stack([np.sort(rng.choice(200, n_si, replace=False)) for _ in range(rows)]).astype(np.int32)
    row_ks = (rng.integers(0, 4, rows) * sbk).astype(np.int32)
    si = si + (row_ks // sbk)[:, None]
    end = rng.integers(1, n_si * sbk + 1, rows).astype(np.int32)
    end[:3] = [n_si * sbk, k, 5]
    x = bf16_decode(bf16_encode(rng.standard_normal((rows, n_si * sbk)).astype(np.float32)))
    x[np.arange(n_si * sbk)[None, :] >= end[:, None]] = -np.inf
    bt = rng.permutation(rows * 256).astype(np.int32).reshape(rows, 256)
    pos = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    cols = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    slots = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    idx.idx_sparse_topk_remap(dev_bf16(bf16_encode(x)), dev(end), dev(si), dev(row_ks), sbk, k, pos,
                              col_scratch=cols, slots=slots, block_table=dev(bt), block_size=64, block_span=64)
    idx.idx_device_error()
    pos, cols, slots = pos.cpu().numpy(), cols.cpu().numpy(), slots.cpu().numpy()
    for r in range(rows):
        e = int(end[r])
        assert_topk_values_exact(cols[r], x[r, :e], k, f"row {r}")
        m = min(k, e)
        assert np.array_equal(pos[r, :m], O.sparse_remap_columns(cols[r, :m], si[r], int(row_ks[r]), sbk))
        assert np.all(pos[r, m:] == -1) and np.all(cols[r, m:] == -1)
        assert slots[r].tolist() == [_slots_closed_form(int(v), bt, r, 64, 64) for v in pos[r]]


@pytest.mark.parametrize("bf16,ld_extra,offset", [(False, 0, 0), (False, 3, 0), (False, 0, 2),
                                                  (True, 0, 0), (True, 5, 0), (True, 0, 1)])
def test_sparse_remap_short_rows_load_paths_and_digit_ties(bf16, ld_extra, offset):
    # many sparse rows of at most 4096 columns: 16-byte loads (aligned rows) and
    # element loads (ld or base not 16-byte aligned), keys equal in every digit but
    # the last (fp32: 4 levels), many keys equal to the threshold key, and the
    # workspace, which these rows never need and the selection only clears
    rows, sbk, k, n_si = 320, 64, 1000, 32
    width = n_si * sbk
    ld = width + ld_extra
    rng = np.random.default_rng(1000 + 10 * ld_extra + offset + bf16)
    si = np.stack([rng.permutation(4 * n_si)[:n_si] for _ in range(rows)]).astype(np.int32)
    end = rng.integers(k - 50, width + 1, rows).astype(np.int32)
    end[:4] = [width, k, k + 1, width - 1]
    x = rng.standard_normal((rows, width)).astype(np.float32)
    x[4::3] = (1.0 + rng.integers(0, 64, (len(range(4, rows, 3)), width)) * 2.0 ** -23).astype(np.float32)
    x[5::3] = rng.integers(-4, 4, (len(range(5, rows, 3)), width)).astype(np.float32) * 0.5
    x[6, :] = 0.75
    x[7, ::7] = -np.inf
    if bf16:
        xb = bf16_encode(x)
        vals = bf16_decode(xb)
        flat = torch.empty(rows * ld + offset, dtype=torch.int16, device=DEV)
        full = np.zeros((rows, ld), dtype=np.uint16)
        full[:, :width] = xb
        flat[offset:] = torch.from_numpy(full.reshape(-1).view(np.int16)).to(DEV)
        t = flat[offset:].view(rows, ld).view(torch.bfloat16)
    else:
        vals = x
        flat = torch.empty(rows * ld + offset, dtype=torch.float32, device=DEV)
        full = np.zeros((rows, ld), dtype=np.float32)
        full[:, :width] = x
        flat[offset:] = torch.from_numpy(full.reshape(-1)).to(DEV)
        t = flat[offset:].view(rows, ld)
    keys = _keys(vals.astype(np.float32).view(np.uint32))
    h = np.zeros((rows, 1024), dtype=np.int32)
    for r in range(rows):
        np.add.at(h[r], (keys[r, :end[r]] >> 22).astype(np.int64), 1)
    ws = dev(h)
    assert idx.idx_workspace_bytes("sparse_topk_remap", rows, ld, k) == 0
    assert idx.idx_workspace_bytes("sparse_topk_remap", 8, ld, k) == 0     # fewer rows than SMs too
    assert idx.idx_workspace_bytes("sparse_topk_remap", rows, 0, k) == rows * 1024 * 4
    pos = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    cols = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    idx.idx_sparse_topk_remap(t, dev(end), dev(si), None, sbk, k, pos, col_scratch=cols, ws=ws)
    idx.idx_device_error()
    assert not ws.any().item(), "the selection hands the workspace back zeroed"
    pos, cols = pos.cpu().numpy(), cols.cpu().numpy()
    for r in range(rows):
        e = int(end[r])
        assert_topk_values_exact(cols[r], vals[r, :e], k, f"row {r}")
        m = min(k, e)
        assert len(set(cols[r, :m].tolist())) == m
        assert np.array_equal(pos[r, :m], O.sparse_remap_columns(cols[r, :m], si[r], 0, sbk))
        assert np.all(pos[r, m:] == -1) and np.all(cols[r, m:] == -1)


def test_topk_ties_overflow_and_special_values():
    width, k = 40000, 2048
    x = W.make_logits(9, 6, width, ties=True)
    x[1, :] = 0.5                                     # all equal: every bucket ties
    x[2, :] = (1.0 + np.arange(width) * 2.0 ** -22).astype(np.float32)  # one top-11-bit bucket
    x[3, ::3] = -np.inf                               # -inf never beats a finite score
    x[4, :30000] = 0.25                               # bucket A overflows, B holds the rest
    x[4, 30000:] = (0.25 + np.arange(10000) * 2.0 ** -24).astype(np.float32)
    x[5, :] = np.float32(-3.0)
    x[5, 123] = np.float32(3.0)
    out, vals = _run_topk(x, None, np.full(6, width, dtype=np.int32), k)
    for r in range(6):
        assert_topk_values_exact(out[r], vals[r], k, f"row {r}")
    assert 123 in set(out[5].tolist())


def _keys(bits_u32):
    """The selection's order-preserving keys of fp32 bit patterns (NaN above +inf, -NaN below -inf)."""
    u = np.asarray(bits_u32, dtype=np.uint32)
    return u ^ (((u.view(np.int32) >> 31).view(np.uint32)) | np.uint32(0x80000000))


@pytest.mark.parametrize("bf16", [False, True])
def test_topk_key_order_special_values_both_compare_paths(bf16):
    # the level-0 hit test compares raw bit patterns when the threshold is a
    # non-negative value and keys otherwise: rows with positive and with negative
    # thresholds, NaNs of both signs, infinities and signed zeros, checked in the
    # key order itself (the selected keys are the k largest keys)
    width, k = 20000, 1000
    rng = np.random.default_rng(77 + bf16)
    x = rng.standard_normal((6, width)).astype(np.float32)
    x[1] -= 10.0                                   # every value negative: a negative threshold
    x[2] = -np.abs(x[2]) - 1.0
    x[2, 5000:5600] = -0.5                         # the threshold sits in a negative tied bucket
    for r in (0, 1, 3):
        x[r, 11] = np.float32(np.nan)              # positive NaN: above +inf
        x[r, 12] = -np.float32(np.nan)             # negative NaN: below -inf
        x[r, 13] = np.float32(np.inf)
        x[r, 14] = -np.float32(np.inf)
        x[r, 15] = np.float32(0.0)
        x[r, 16] = -np.float32(0.0)
    x[3, :] = np.abs(x[3]) * 1e-30                 # tiny positive values, subnormal keys
    x[4, ::2] = 0.0
    x[4, 1::2] = -0.0                              # only signed zeros
    x[5, :] = -np.float32(np.nan)
    x[5, 100:3000] = rng.standard_normal(2900).astype(np.float32)
    if bf16:
        xb = bf16_encode(np.where(np.isnan(x), 0, x))
        sign = np.signbit(x) & np.isnan(x)
        xb = np.where(np.isnan(x), np.where(sign, 0xFFC0, 0x7FC0), xb).astype(np.uint16)
        t = dev_bf16(xb)
        bits = xb.astype(np.uint32) << 16
    else:
        t = dev(x)
        bits = x.view(np.uint32)
    out = torch.full((6, k), -7, dtype=torch.int32, device=DEV)
    idx.idx_topk(t, None, dev(np.full(6, width, dtype=np.int32)), k, out)
    o = out.cpu().numpy()
    for r in range(6):
        keys = _keys(bits[r])
        assert len(np.unique(o[r])) == k and np.all((o[r] >= 0) & (o[r] < width)), f"row {r}"
        want = np.sort(keys)[::-1][:k]
        got = np.sort(keys[o[r]])[::-1]
        assert np.array_equal(got, want), f"row {r}: selected keys differ from the {k} largest keys"
    assert 11 in set(o[0].tolist()) and 12 not in set(o[0].tolist())


def test_topk_bf16_and_wide_rows():
    x = W.make_logits(10, 4, 131072)
    out, vals = _run_topk(x, None, np.full(4, 131072, dtype=np.int32), 2048, bf16=True)
    for r in range(4):
        assert_topk_values_exact(out[r], vals[r], 2048, f"bf16 row {r}")
    out, vals = _run_topk(x, None, np.array([131072, 65536, 2048, 0], dtype=np.int32), 2048)
    for r in range(4):
        n = [131072, 65536, 2048, 0][r]
        assert_topk_values_exact(out[r], vals[r, :n], 2048, f"fp32 row {r}")
        ref = O.topk_row(vals[r], 0, n, 2048)
        assert set(out[r].tolist()) == set(ref.tolist())


@pytest.mark.parametrize("bf16", [False, True])
def test_topk_more_rows_than_sms(bf16):
    # more rows than SMs: blocks run in waves and each asks for the row one wave
    # ahead to be staged in L2; ragged causal ranges, odd row stride, empty rows
    rows, width, k = 700, 6000, 512
    x = W.make_logits(31 + bf16, rows, width, ties=True)
    rng = np.random.default_rng(31)
    ks = rng.integers(0, 1500, rows).astype(np.int32)
    ke = np.minimum(ks + rng.integers(0, width, rows), width).astype(np.int32)
    ke[5], ks[5] = 0, 0                       # empty row
    ke[6] = ks[6] + 300                       # fewer visible columns than k
    out, vals = _run_topk(x, ks, ke, k, bf16=bf16, ld_pad=3)
    for r in range(rows):
        seg = vals[r, ks[r]:ke[r]]
        assert_topk_values_exact(out[r], seg, k, f"row {r}")
        if r % 50 == 0 and len(np.unique(seg)) == len(seg):
            assert set(out[r].tolist()) == set(O.topk_row(vals[r], ks[r], ke[r], k).tolist())


def test_topk_more_rows_than_sms_ties_and_overflow():
    # the two-blocks-per-SM configuration (many rows, at most 64K columns) with the
    # rows that overflow its smaller buckets and force the global re-read paths
    rows, width, k = 400, 40000, 2048
    x = W.make_logits(33, rows, width, ties=True)
    x[1::8, :] = 0.5                                                  # every bucket ties
    x[2::8, :] = (1.0 + np.arange(width) * 2.0 ** -22).astype(np.float32)  # one first-digit bucket
    x[3::8, ::3] = -np.inf
    x[4::8, :30000] = 0.25                                            # level-0 bucket overflows
    x[4::8, 30000:] = (0.25 + np.arange(10000) * 2.0 ** -24).astype(np.float32)
    x[5::8, :] = np.float32(-3.0)
    x[5::8, 123] = np.float32(3.0)
    ke = np.full(rows, width, dtype=np.int32)
    ke[6::8] = 1000                                                   # fewer columns than k
    out, vals = _run_topk(x, None, ke, k)
    for r in range(rows):
        assert_topk_values_exact(out[r], vals[r, :ke[r]], k, f"row {r}")
    assert all(123 in set(out[r].tolist()) for r in range(5, rows, 8))


@pytest.mark.parametrize("bf16", [False, True])
def test_topk_values_output(bf16):
    # the optional score output: the score of every selected column, -inf in -1 slots
    width, k = 9000, 2048
    x = W.make_logits(13, 5, width, ties=True)
    ke = np.array([width, 5000, 2048, 100, 0], dtype=np.int32)
    if bf16:
        xb = bf16_encode(x)
        t, vals = dev_bf16(xb), bf16_decode(xb)
    else:
        t, vals = dev(x), x
    out = torch.full((5, k + 3), -7, dtype=torch.int32, device=DEV)
    sc = torch.full((5, k + 1), 7.0, dtype=torch.float32, device=DEV)
    idx.idx_topk(t, None, dev(ke), k, out, vals=sc[:, :k + 1])
    o, v = out.cpu().numpy(), sc.cpu().numpy()
    for r in range(5):
        n = int(ke[r])
        m = min(n, k)
        assert_topk_values_exact(o[r], vals[r, :n], k, f"row {r}")
        assert np.array_equal(v[r, :m], vals[r, o[r, :m]].astype(np.float32)), f"scores row {r}"
        assert np.all(np.isneginf(v[r, m:k])) and v[r, k] == 7.0


def _oracle_candidates(row, bounds, k_local):
    """Each shard's local top-k by the oracle: (values, shard-local indices), -inf / -1 padded."""
    n_shards = len(bounds) - 1
    cv = np.full(n_shards * k_local, -np.inf, dtype=np.float32)
    ci = np.full(n_shards * k_local, -1, dtype=np.int32)
    for s in range(n_shards):
        loc = O.topk_row(row, int(bounds[s]), int(bounds[s + 1]), k_local)
        ok = loc >= 0
        ci[s * k_local:(s + 1) * k_local] = loc
        cv[s * k_local:(s + 1) * k_local][ok] = row[bounds[s] + loc[ok]]
    return cv, ci


def _check_merge(pos, v, cand_pos, cand_val, k, what):
    """Merged output against the oracle's merge of the same candidates: the value
    multiset is unique; each position must be a distinct candidate with its value."""
    ref_p, ref_v = O.dcp_topk_merge_row(cand_val, cand_pos, None, len(cand_pos), k)
    m = int(np.sum(ref_p >= 0))
    assert np.all(pos[m:k] == -1) and np.all(np.isneginf(v[m:k])), f"{what}: tail"
    assert len(np.unique(pos[:m])) == m and np.all(pos[:m] >= 0), f"{what}: positions"
    assert np.array_equal(np.sort(v[:m].astype(np.float64))[::-1], ref_v[:m]), f"{what}: values"
    lut = {}
    for p_, v_ in zip(cand_pos.tolist(), cand_val.tolist()):
        if p_ >= 0:
            lut[p_] = v_
    assert all(lut.get(int(p_)) == float(v_) for p_, v_ in zip(pos[:m], v[:m])), f"{what}: pairs"


def _shard_candidates(x_row, n, n_shards, k_local, mode, rng):
    """Oracle local top-k of one row's shards: (values, local indices, offsets, stride)."""
    if mode == "interleaved":            # token t lives on shard t % n_shards
        cv = np.full(n_shards * k_local, -np.inf, dtype=np.float32)
        ci = np.full(n_shards * k_local, -1, dtype=np.int32)
        for s in range(n_shards):
            loc_row = x_row[s:n:n_shards]
            loc = O.topk_row(loc_row, 0, len(loc_row), k_local)
            ok = loc >= 0
            ci[s * k_local:(s + 1) * k_local] = loc
            cv[s * k_local:(s + 1) * k_local][ok] = loc_row[loc[ok]]
        return cv, ci, np.arange(n_shards, dtype=np.int32), n_shards
    cuts = np.sort(rng.integers(0, n + 1, n_shards - 1))
    b = np.concatenate([[0], cuts, [n]]).astype(np.int64)
    cv, ci = _oracle_candidates(x_row, b, k_local)
    return cv, ci, b[:-1].astype(np.int32), 1


@pytest.mark.parametrize("mode", ["per_row", "interleaved"])
@pytest.mark.parametrize("n_shards,k_local,k", [(2, 2048, 2048), (8, 2048, 2048), (3, 700, 2048),
                                                (4, 512, 1000), (1, 100, 64), (5, 300, 4096)])
def test_dcp_merge_vs_oracle(n_shards, k_local, k, mode):
    # candidates from the oracle's local top-k of seeded rows (ties included),
    # merged by the library and by the oracle
    rows, width = 6, 20000
    x = W.make_logits(14 + n_shards, rows, width, ties=True)
    x[1] = np.float32(0.5)                                  # every candidate ties
    rng = np.random.default_rng(n_shards * 1000 + k_local)
    lens = rng.integers(0, width + 1, rows)
    lens[0], lens[2] = width, 37                            # full row; fewer candidates than k
    cv = np.zeros((rows, n_shards * k_local), dtype=np.float32)
    ci = np.zeros((rows, n_shards * k_local), dtype=np.int32)
    offs = np.zeros((rows, n_shards), dtype=np.int32)
    for r in range(rows):
        cv[r], ci[r], offs[r], stride = _shard_candidates(x[r], int(lens[r]), n_shards, k_local, mode, rng)
    d_offs = dev(offs[0]) if mode == "interleaved" else dev(offs)   # shared vector / one per row
    out = torch.full((rows, k + 2), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((rows, k), dtype=torch.float32, device=DEV)
    idx.idx_dcp_topk_merge(dev(cv), dev(ci), d_offs, k_local, k, out, vals=sc, pos_stride=stride)
    o, v = out.cpu().numpy(), sc.cpu().numpy()
    assert np.all(o[:, k:] == -7)
    gpos = np.where(ci >= 0, offs.repeat(k_local, axis=1) + ci * stride, -1).astype(np.int32)
    for r in range(rows):
        _check_merge(o[r], v[r], gpos[r], cv[r], k, f"row {r}")
        ref_p, _ = O.dcp_topk_merge_row(cv[r], ci[r], offs[r], k_local, k, stride)
        m = int(np.sum(ref_p >= 0))
        if len(np.unique(cv[r][ci[r] >= 0])) == int(np.sum(ci[r] >= 0)):   # no ties: unique set
            assert set(o[r, :m].tolist()) == set(ref_p[:m].tolist())
    # indices already global: the same selection without offsets
    out2 = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    idx.idx_dcp_topk_merge(dev(cv), dev(gpos), None, k_local, k, out2)
    o2 = out2.cpu().numpy()
    for r in range(rows):
        lut = dict(zip(gpos[r].tolist(), cv[r].tolist()))
        v2 = np.array([lut[p_] if p_ >= 0 else -np.inf for p_ in o2[r].tolist()], dtype=np.float32)
        _check_merge(o2[r], v2, gpos[r], cv[r], k, f"global-index row {r}")


@pytest.mark.parametrize("n_shards", [2, 4, 8])
def test_dcp_emulated_ranks_equal_whole_row_topk(n_shards):
    # Every rank selects within its own shard of the row on the device (top-k with
    # scores, written straight into its part of the exchange buffer); the merge of
    # the exchanged lists is the whole row's top-k.
    rows, width, k = 6, 131072, 2048
    x = W.make_logits(20 + n_shards, rows, width, ties=n_shards == 4)
    x[3, ::2] = np.float32(1.0)                             # 65536 equal top scores
    lens = np.array([width, 100000, 3000, width, 2048 * n_shards, 1], dtype=np.int64)
    bounds = np.linspace(0, width, n_shards + 1).astype(np.int64)
    bounds[1:-1] = bounds[1:-1] // 16 * 16 + 3              # ragged, unaligned shard starts
    t = dev(x)
    cv = torch.empty((rows, n_shards * k), dtype=torch.float32, device=DEV)
    ci = torch.empty((rows, n_shards * k), dtype=torch.int32, device=DEV)
    for s in range(n_shards):
        lo, hi = int(bounds[s]), int(bounds[s + 1])
        ke = np.clip(lens - lo, 0, hi - lo).astype(np.int32)
        idx.idx_topk(t[:, lo:], None, dev(ke), k, ci[:, s * k:(s + 1) * k],
                     vals=cv[:, s * k:(s + 1) * k])
    out = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    sc = torch.empty((rows, k), dtype=torch.float32, device=DEV)
    idx.idx_dcp_topk_merge(cv, ci, dev(bounds[:-1].astype(np.int32)), k, k, out, vals=sc)
    o, v = out.cpu().numpy(), sc.cpu().numpy()
    for r in range(rows):
        n = int(lens[r])
        assert_topk_values_exact(o[r], x[r, :n], k, f"row {r}")
        m = min(n, k)
        assert np.array_equal(v[r, :m], x[r, o[r, :m]]), f"scores row {r}"
        if len(np.unique(x[r, :n])) == n:
            assert set(o[r, :m].tolist()) == set(O.topk_row(x[r], 0, n, k)[:m].tolist())


def test_dcp_merge_degenerate():
    # all candidates empty; a single candidate; zero rows; bad strides
    k_local, k = 16, 8
    cv = np.full((3, 2 * k_local), -np.inf, dtype=np.float32)
    ci = np.full((3, 2 * k_local), -1, dtype=np.int32)
    cv[1, 20], ci[1, 20] = 2.5, 9
    cv[2, :] = np.arange(2 * k_local, dtype=np.float32)
    ci[2, :] = np.arange(2 * k_local)
    out = torch.full((3, k), -7, dtype=torch.int32, device=DEV)
    idx.idx_dcp_topk_merge(dev(cv), dev(ci), dev(np.array([0, 1000], dtype=np.int32)), k_local, k, out)
    o = out.cpu().numpy()
    assert np.all(o[0] == -1)
    assert o[1].tolist() == [1000 + 9] + [-1] * (k - 1)
    assert sorted(o[2].tolist()) == [1000 + j for j in range(24, 32)]
    empty = torch.empty((0, k), dtype=torch.int32, device=DEV)
    idx.idx_dcp_topk_merge(dev(cv[:0]), dev(ci[:0]), None, k_local, k, empty)
    with pytest.raises(idx.IdxError):
        idx.idx_dcp_topk_merge(dev(cv), dev(ci), None, 64, k, out)


def test_k_quant_rounding_boundaries():
    # Values whose quotient by the token scale sits on, or a few ulps either side
    # of, every e4m3 rounding midpoint, for scales that are and are not powers of
    # two: the bytes must equal the oracle's division-per-element definition.
    codes = e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64)   # 0 .. 448
    mids = (codes[:-1] + codes[1:]) / 2.0

    def steps(x, d):
        x = np.float32(x)
        to = np.float32(np.inf) if d > 0 else np.float32(-np.inf)
        for _ in range(abs(d)):
            x = np.nextafter(x, to)
        return x

    rows = []
    for amax in (448.0, 300.0, 1.0, 3.0e-3, 123.456, 7.0e-5):
        s = np.float32(np.float32(amax) / np.float32(448.0))
        for sign in (1.0, -1.0):
            vals = [np.float32(sign) * steps(np.float32(m) * s, d) for m in mids for d in range(-4, 5)]
            vals = np.array(vals, dtype=np.float32)
            for a in range(0, len(vals), 127):
                row = np.zeros(128, dtype=np.float32)
                row[0] = np.float32(amax)
                chunk = vals[a:a + 127]
                chunk = chunk[np.abs(chunk) <= np.float32(amax)]
                row[1:1 + len(chunk)] = chunk
                rows.append(row)
    k = np.stack(rows)
    n = len(k)
    slots = np.arange(n, dtype=np.int64)
    bs = 64
    nblk = (n + bs - 1) // bs
    stride = W.block_stride_bytes(bs)
    gcache = torch.zeros((nblk, stride), dtype=torch.uint8, device=DEV)
    idx.idx_k_quant_and_cache(dev(k), dev(slots), gcache, bs)
    ocache = np.zeros((nblk, stride), dtype=np.uint8)
    O.k_quant_and_cache(k, slots, ocache, bs)
    assert np.array_equal(gcache.cpu().numpy(), ocache)


# ------------------------------------------------------------------ q preparation

def _cos_sin(max_pos, base=10000.0):
    i = np.arange(32, dtype=np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * base ** (-2.0 * i / 64.0)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


@pytest.mark.parametrize("T", [1, 37, 300])
@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("q_bf16,w_bf16,out_bf16", [(True, False, False), (True, True, True),
                                                    (False, False, True)])
def test_q_rope_quant_vs_oracle(T, interleaved, q_bf16, w_bf16, out_bf16):
    rng = np.random.default_rng(T * 7 + interleaved)
    max_pos = 5000
    qf = (rng.standard_normal((T, 64, 128)) * rng.uniform(0.01, 30, (T, 64, 1))).astype(np.float32)
    qf[0, 3] = 0.0                                        # an all-zero head: scale 0
    wf = rng.standard_normal((T, 64)).astype(np.float32)
    pos = rng.integers(0, max_pos, T).astype(np.int32)
    cs = np.zeros((max_pos, 72), dtype=np.float32)        # strided table
    cs[:, :64] = _cos_sin(max_pos)
    pad = 64                                              # strided q rows (elements)
    if q_bf16:
        qb = bf16_encode(qf)
        qv = bf16_decode(qb).astype(np.float32)
        buf = np.zeros((T, 8192 + pad), dtype=np.uint16)
        buf[:, :8192] = qb.reshape(T, -1)
        q_dev = dev_bf16(buf)[:, :8192]
    else:
        qv = qf
        buf = np.zeros((T, 8192 + pad), dtype=np.float32)
        buf[:, :8192] = qf.reshape(T, -1)
        q_dev = dev(buf)[:, :8192]
    if w_bf16:
        wb = bf16_encode(wf)
        wv, w_dev = bf16_decode(wb).astype(np.float32), dev_bf16(wb)
    else:
        wv, w_dev = wf, dev(wf)
    q8 = torch.full((T, 8192 + 32), 7, dtype=torch.uint8, device=DEV)
    w_out = torch.empty((T, 64), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=DEV)
    ss, nhs = 128 ** -0.5, 64 ** -0.5
    idx.idx_q_rope_quant(q_dev, dev(pos), dev(cs)[:, :], w_dev, q8[:, :8192], w_out, ss, nhs, interleaved)
    idx.idx_device_error()
    o8, ow, _ = O.q_rope_quant(qv.reshape(T, 64, 128), pos, cs[:, :64], wv, ss, nhs, interleaved)
    g8 = q8.cpu().numpy()
    assert np.array_equal(g8[:, :8192].reshape(T, 64, 128), o8), "q8 bytes"
    assert np.all(g8[:, 8192:] == 7), "bytes past the row must stay untouched"
    if out_bf16:
        assert np.array_equal(host_bf16(w_out), bf16_encode(ow)), "bf16 weights"
    else:
        assert np.array_equal(w_out.cpu().numpy(), ow), "fp32 weights"


def test_q_rope_quant_flags_bad_positions():
    T = 4
    q = dev_bf16(bf16_encode(np.ones((T, 8192), dtype=np.float32)))
    w = dev(np.ones((T, 64), dtype=np.float32))
    q8 = torch.empty((T, 8192), dtype=torch.uint8, device=DEV)
    w_out = torch.empty((T, 64), dtype=torch.float32, device=DEV)
    cs = dev(_cos_sin(8))
    idx.idx_q_rope_quant(q, dev(np.array([0, 8, -1, 7], dtype=np.int32)), cs, w, q8, w_out, 1.0, 1.0)
    with pytest.raises(idx.IdxError, match="q rope 0x00000001"):
        idx.idx_device_error()
    g = q8.cpu().numpy()
    assert np.all(g[1] == 0) and np.all(g[2] == 0) and g[0].any() and g[3].any()
    assert np.all(w_out.cpu().numpy()[1:3] == 0)
    idx.idx_device_error()                                 # the flag was cleared


# ------------------------------------------------------------------ a7 expansion, a6 slots

def test_expand_candidates_random_vs_oracle():
    rng = np.random.default_rng(12)
    for sbk, R, K in [(64, 1, 64), (8, 2, 16), (16, 4, 32), (8, 8, 128), (64, 1, 1024), (32, 2, 2)]:
        rows = 37
        cbs = sbk * R
        ks = (rng.integers(0, 50, rows) * sbk).astype(np.int32)
        ke = (ks + rng.integers(0, 40 * cbs, rows)).astype(np.int32)
        cand = rng.integers(-2, 45, (rows, K + 3)).astype(np.int32)   # ld_c = K + 3
        gsi = torch.full((rows, K * R + 2), -9, dtype=torch.int32, device=DEV)
        gend = torch.empty(rows, dtype=torch.int32, device=DEV)
        idx.idx_expand_candidates(dev(cand)[:, :K], dev(ks), dev(ke), cbs, sbk, gsi[:, :K * R], gend)
        osi, oend = O.expand_candidates(cand[:, :K], ks, ke, cbs, sbk)
        s = gsi.cpu().numpy()
        assert np.array_equal(s[:, :K * R], osi), (sbk, R, K)
        assert np.all(s[:, K * R:] == -9)
        assert np.array_equal(gend.cpu().numpy(), oend), (sbk, R, K)


def test_expand_candidates_golden():
    import json
    import os

    with open(os.path.join(os.path.dirname(__file__), "golden", "expand_candidates.json")) as f:
        spec = json.load(f)
    for c in spec["cases"]:
        cand = np.array([c["cand"]], dtype=np.int32)
        si = torch.empty((1, len(c["sparse_idx"])), dtype=torch.int32, device=DEV)
        end = torch.empty(1, dtype=torch.int32, device=DEV)
        idx.idx_expand_candidates(dev(cand), dev(np.array([c["ks"]], np.int32)),
                                  dev(np.array([c["ke"]], np.int32)), c["cand_block_size"], c["sbk"],
                                  si, end)
        assert si.cpu().numpy()[0].tolist() == c["sparse_idx"], c["note"]
        assert int(end.cpu()[0]) == c["end"], c["note"]


def test_expand_candidates_flags_misaligned_ks():
    cand = dev(np.array([[0, 1, 2, 3]], dtype=np.int32))
    si = torch.empty((1, 4), dtype=torch.int32, device=DEV)
    end = torch.empty(1, dtype=torch.int32, device=DEV)
    idx.idx_expand_candidates(cand, dev(np.array([10], np.int32)), dev(np.array([500], np.int32)),
                              64, 64, si, end)
    with pytest.raises(idx.IdxError):
        idx.idx_device_error()
    assert int(end.cpu()[0]) == 0
    idx.idx_device_error()   # the flag was cleared


def test_req_to_global_slots_vs_oracle():
    import json
    import os

    with open(os.path.join(os.path.dirname(__file__), "golden", "slot_remap.json")) as f:
        spec = json.load(f)
    bt = np.array([spec["block_table"]], dtype=np.int32)
    for c in spec["cases"]:
        loc = dev(np.array([[c["local"]]], dtype=np.int32))
        out = torch.empty_like(loc)
        idx.idx_req_to_global_slots(loc, None, dev(bt), spec["block_size"], c["block_span"], out)
        assert int(out.cpu()[0, 0]) == c["slot"]
    rng = np.random.default_rng(3)
    rows, k, nreq = 50, 2048, 7
    bt = rng.integers(0, 5000, (nreq, 300)).astype(np.int32)
    r2r = rng.integers(0, nreq, rows).astype(np.int32)
    local = rng.integers(-1, 300 * 64, (rows, k)).astype(np.int32)
    for span in (64, 68, 80):
        out = torch.empty((rows, k + 1), dtype=torch.int32, device=DEV)
        idx.idx_req_to_global_slots(dev(local), dev(r2r), dev(bt), 64, span, out[:, :k])
        ref = O.req_to_global_slots(local, r2r, bt, 64, span)
        assert np.array_equal(out.cpu().numpy()[:, :k], ref)
    g = dev(local)                                     # in place
    idx.idx_req_to_global_slots(g, dev(r2r), dev(bt), 64, 64, g)
    assert np.array_equal(g.cpu().numpy(), O.req_to_global_slots(local, r2r, bt, 64, 64))


def test_sparse_topk_remap_vs_oracle_bf16():
    rows, n_si, sbk, k = 9, 64, 64, 2048
    x = W.make_logits(20, rows, n_si * sbk)
    xb = bf16_encode(x)
    rng = np.random.default_rng(20)
    si = np.sort(rng.choice(4000, (rows, n_si)), axis=1).astype(np.int32)
    end = np.array([4096, 4000, 2048, 2047, 100, 0, 1, 3000, 4096], dtype=np.int32)
    pos = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    cols = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    idx.idx_sparse_topk_remap(dev_bf16(xb), dev(end), dev(si), None, sbk, k, pos, col_scratch=cols)
    pos, cols = pos.cpu().numpy(), cols.cpu().numpy()
    vals = bf16_decode(xb)
    for r in range(rows):
        e = int(end[r])
        assert_topk_values_exact(cols[r], vals[r, :e], k, f"row {r}")
        m = min(k, e)
        expect = [(int(si[r, c // sbk])) * sbk + c % sbk for c in cols[r, :m]]
        assert pos[r, :m].tolist() == expect and np.all(pos[r, m:] == -1)


# ------------------------------------------------------------------ selection workspace

def _first_digit_hist(vals_f32):
    u = np.ascontiguousarray(vals_f32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    key = np.where(u & 0x80000000, ~u & 0xFFFFFFFF, u | 0x80000000)
    return np.bincount((key >> 22).astype(np.int64), minlength=1024)


def test_selection_workspace_dense_decode():
    ctx = np.array([1000, 2048, 3000, 4096, 5000, 1, 2049, 300], dtype=np.int32)
    pool = W.make_pool(55, ctx)
    g, o = build_caches(pool, 55)
    q8, w = W.make_q(56, len(ctx))
    rows = len(ctx)
    ld = (int(ctx.max()) + 63) // 64 * 64
    out = torch.empty((rows, ld), dtype=torch.float32, device=DEV)
    ws = torch.zeros((rows, 1024), dtype=torch.int32, device=DEV)
    idx.idx_paged_mqa_logits_decode(dev(q8), dev(w), g, 64, dev(pool.block_table), dev(ctx), out, ws=ws)
    lg = out.cpu().numpy()
    hist = ws.cpu().numpy()
    for r in range(rows):   # the histogram describes exactly the visible scores written
        assert np.array_equal(hist[r], _first_digit_hist(lg[r, :ctx[r]])), r
    k = 2048
    a = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    b = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    idx.idx_topk(out, None, dev(ctx), k, a, ws=ws)
    assert not ws.any().item(), "the selection hands the workspace back zeroed"
    idx.idx_topk(out, None, dev(ctx), k, b)
    a, b = a.cpu().numpy(), b.cpu().numpy()
    ref = O.paged_decode_logits(q8, w, o, 64, pool.block_table, ctx, 1)
    for r in range(rows):
        assert_topk_values_exact(a[r], lg[r, :ctx[r]], k, f"ws row {r}")
        assert np.array_equal(np.sort(lg[r, a[r][a[r] >= 0]]), np.sort(lg[r, b[r][b[r] >= 0]]))
        assert_topk_row(a[r], ref[r, :ctx[r]], k, f"ws vs oracle row {r}")


def test_selection_workspace_sparse_paths():
    ctx, pool, g, o, q8, w, cand = _hier_inputs(71)
    rows = len(ctx)
    si = torch.empty((rows, 16), dtype=torch.int32, device=DEV)
    end = torch.empty(rows, dtype=torch.int32, device=DEV)
    idx.idx_expand_candidates(dev(cand), None, dev(ctx), 64, 64, si, end)
    out = torch.empty((rows, 1024), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros((rows, 1024), dtype=torch.int32, device=DEV)
    idx.idx_paged_mqa_logits_decode(dev(q8), dev(w), g, 64, dev(pool.block_table), dev(ctx), out,
                                    sparse_idx=si, end=end, sbk=64, ws=ws)
    lg = out.float().cpu().numpy()
    e = end.cpu().numpy()
    hist = ws.cpu().numpy()
    for r in range(rows):
        assert np.array_equal(hist[r], _first_digit_hist(lg[r, :e[r]])), r
    k = 300
    pa = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    pb = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    ca = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    cb = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    idx.idx_sparse_topk_remap(out, end, si, None, 64, k, pa, col_scratch=ca, ws=ws)
    assert not ws.any().item()
    idx.idx_sparse_topk_remap(out, end, si, None, 64, k, pb, col_scratch=cb)
    ca, cb, pa, pb = ca.cpu().numpy(), cb.cpu().numpy(), pa.cpu().numpy(), pb.cpu().numpy()
    sih = si.cpu().numpy()
    for r in range(rows):
        assert_topk_values_exact(ca[r], lg[r, :e[r]], k, f"sparse ws row {r}")
        # with or without the fused histogram: the same multiset of chosen scores,
        # and every position is its column's token
        m = min(k, int(e[r]))
        assert np.array_equal(np.sort(lg[r, ca[r, :m]]), np.sort(lg[r, cb[r, :m]])), r
        for c_, p_ in ((ca, pa), (cb, pb)):
            assert [O.sparse_column_token(sih[r], int(c), 64) for c in c_[r, :m]] == p_[r, :m].tolist(), r
            assert np.all(p_[r, m:] == -1), r
    # dense prefill runs four queries per group: the workspace is refused there
    k8, ks = W.make_random_cache_tokens(3, 256)
    q2, w2 = W.make_q(4, 8)
    lo = torch.empty((8, 256), dtype=torch.float32, device=DEV)
    with pytest.raises(idx.IdxError):
        idx.idx_mqa_logits_prefill(dev(q2), dev(w2), dev(k8), dev(ks), None,
                                   dev(np.full(8, 256, np.int32)), lo,
                                   ws=torch.zeros((8, 1024), dtype=torch.int32, device=DEV))


def test_diag_l2_read_rate_is_plausible():
    # the L2 read-rate diagnostic: a 64 MB buffer (inside L2) read by every SM;
    # the rate must lie between the HBM copy rate's order and far below any
    # physical limit (a dropped load would show as an absurd rate)
    import bench

    r = bench.measure_l2_read(mb=64, passes=10)
    idx.idx_device_error()
    assert 1000.0 < r["gbs"] < 100000.0, r
