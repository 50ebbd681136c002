"""Parity of the MXFP4 indexer cache path with the CPU oracle.

The insert must reproduce the oracle's cache bytes bit for bit (the OCP MX
conversion: every e2m1 rounding tie, saturation, the clamped exponent range);
the fp8 x fp4 scores must match the oracle within 1e-3 + 2e-3 * |oracle| over
every block size, ragged contexts and both output types, in the dense and the
sparse (V4.1 hierarchical) modes; selections are checked against the oracle up
to ties and exactly against the scores the kernel wrote.
"""

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


def build_mx_caches(pool, seed, block_size=64, stride=None):
    """MXFP4 cache filled by the kernel and by the oracle from the same bf16 k."""
    stride = stride or W.mxfp4_block_stride_bytes(block_size)
    g = torch.zeros((pool.num_blocks, stride), dtype=torch.uint8, device=DEV)
    o = np.zeros((pool.num_blocks, stride), dtype=np.uint8)
    ks = []
    for b in range(len(pool.ctx_lens)):
        kb = W.make_k(seed, b, int(pool.ctx_lens[b]))
        ks.append(kb)
        O.mxfp4_k_quant_and_cache(bf16_decode(kb), pool.slot_mapping(b), o, block_size)
    slots = dev(np.concatenate([pool.slot_mapping(b) for b in range(len(pool.ctx_lens))]))
    idx.idx_k_quant_and_cache_mxfp4(dev_bf16(np.concatenate(ks)), slots, g, block_size)
    return g, o


def _special_tokens():
    """fp32 tokens that hit every rounding tie of e2m1, saturation and the exponent clamps."""
    rng = np.random.default_rng(3)
    toks = []
    for s in (-20, -3, 0, 5, 40):
        t = np.zeros(128, dtype=np.float32)
        scale = np.float32(2.0 ** s)
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
        blk = np.concatenate([[6.0], mids, -mids, [0.0, -0.0, 6.5, 7.99, -7.0]]).astype(np.float32)
        t[:len(blk)] = blk * scale                                # block 0: every tie at amax 6.5 * 2^s
        up = np.nextafter(mids * scale, np.float32(np.inf))
        dn = np.nextafter(mids * scale, np.float32(-np.inf))
        t[32:32 + 7] = up                                          # block 1: just above the ties
        t[39:46] = dn                                              # ... and just below
        t[46] = np.float32(6.0) * scale
        t[64:96] = rng.standard_normal(32).astype(np.float32) * scale   # block 2: random
        toks.append(t)                                             # block 3: all zero
    tiny = np.zeros(128, dtype=np.float32)
    tiny[:32] = np.float32(2.0 ** -130) * rng.standard_normal(32).astype(np.float32)   # subnormal block
    tiny[32:64] = np.float32(1.5 * 2.0 ** 127)                     # the top of the range
    tiny[64] = -np.float32(2.0 ** -149)
    toks.append(tiny)
    return np.stack(toks)


@pytest.mark.parametrize("block_size,f32", [(64, False), (16, True), (128, False), (32, True)])
def test_mxfp4_insert_bitexact(block_size, f32):
    ctx = np.array([300, 1, 65, 1024], dtype=np.int32)
    pool = W.make_pool(91, ctx, block_size=block_size, extra_blocks=3)
    stride = W.mxfp4_block_stride_bytes(block_size)
    g = torch.zeros((pool.num_blocks, stride), dtype=torch.uint8, device=DEV)
    o = np.zeros((pool.num_blocks, stride), dtype=np.uint8)
    k = np.concatenate([bf16_decode(W.make_k(91, b, int(ctx[b]))) for b in range(len(ctx))])
    spec = _special_tokens()
    k[:len(spec)] = spec if f32 else bf16_decode(torch.from_numpy(spec).to(torch.bfloat16).view(torch.int16)
                                                  .numpy().view(np.uint16))
    slots = np.concatenate([pool.slot_mapping(b) for b in range(len(ctx))])
    slots[8] = -1                                                  # skipped: negative ...
    slots[9] = pool.num_blocks * block_size + 3                    # ... or past the pool
    oslots = slots.copy()
    oslots[9] = -1
    O.mxfp4_k_quant_and_cache(k, oslots, o, block_size)
    if f32:
        kd = dev(k.astype(np.float32))
    else:
        kd = dev(k.astype(np.float32)).to(torch.bfloat16)
    # strided input: every token's 128 values inside a wider row
    wide = torch.zeros((k.shape[0], 160), dtype=kd.dtype, device=DEV)
    wide[:, :128] = kd
    idx.idx_k_quant_and_cache_mxfp4(wide[:, :128], dev(slots), g, block_size)
    idx.idx_device_error()
    got = g.cpu().numpy()
    bad = np.nonzero(got != o)
    assert bad[0].size == 0, f"{bad[0].size} bytes differ, first at block {bad[0][:4]}, byte {bad[1][:4]}"


@pytest.mark.parametrize("block_size,out_bf16,w_bf16", [(64, False, False), (16, True, False),
                                                        (32, False, True), (128, True, True)])
def test_mxfp4_decode_dense_logits_and_selection(block_size, out_bf16, w_bf16):
    ctx = np.array([1000, 2048, 3000, 4096, 1, 5, 130, 127, 2049, 64], dtype=np.int32)
    pool = W.make_pool(93, ctx, block_size=block_size, extra_blocks=5)
    g, o = build_mx_caches(pool, 93, block_size)
    rows = len(ctx)
    q8, w = W.make_q(94, rows, w_bf16=w_bf16)
    qbig = np.zeros((rows, 2, 64, 128), dtype=np.uint8)
    qbig[:, 1] = q8
    gq = dev(qbig.reshape(rows, 128, 128))[:, 64:, :]
    gw = dev_bf16(w) if w_bf16 else dev(w)
    L_max = int(ctx.max())
    out = torch.full((rows, L_max + 24), 7.0, device=DEV, dtype=torch.bfloat16 if out_bf16 else torch.float32)
    ws = torch.zeros((rows, 1024), dtype=torch.int32, device=DEV)
    idx.idx_paged_mqa_logits_decode_mxfp4(gq, gw, g, block_size, dev(pool.block_table), dev(ctx), out, ws=ws)
    k = 512
    sel = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    idx.idx_topk(out, None, dev(ctx), k, sel, ws=ws)
    idx.idx_device_error()
    assert not ws.any().item()
    wv = bf16_decode(w) if w_bf16 else w
    ref = O.paged_decode_logits_mxfp4(q8, wv, o, block_size, pool.block_table, ctx)
    got = out.float().cpu().numpy()
    s = sel.cpu().numpy()
    for r in range(rows):
        L = int(ctx[r])
        assert_logits_close(got[r, :L], ref[r, :L], f"row {r}", bf16=out_bf16)
        assert np.all(got[r, L:] == 7.0), "columns beyond the context must stay untouched"
        assert_topk_values_exact(s[r], got[r, :L], k, f"row {r} selection on its own scores")
        assert_topk_row(s[r], ref[r, :L], k, f"row {r} selection vs oracle", bf16=out_bf16)


def test_mxfp4_decode_sparse_hierarchical():
    ctx = np.array([1000, 777, 4096, 2500, 64, 3, 8192, 129], dtype=np.int32)
    pool = W.make_pool(95, ctx)
    g, o = build_mx_caches(pool, 95)
    rows = len(ctx)
    q8, w = W.make_q(96, rows)
    cand = W.make_candidates(97, rows, 16, 40)
    for sbk in (64, 16):
        si = torch.empty((rows, 16 * (64 // sbk)), dtype=torch.int32, device=DEV)
        end = torch.empty(rows, dtype=torch.int32, device=DEV)
        idx.idx_expand_candidates(dev(cand), None, dev(ctx), 64, sbk, si, end)
        osi, oend = O.expand_candidates(cand, None, ctx, 64, sbk)
        assert np.array_equal(si.cpu().numpy(), osi) and np.array_equal(end.cpu().numpy(), oend)
        ncols = si.shape[1] * sbk
        out = torch.empty((rows, ncols), dtype=torch.bfloat16, device=DEV)
        ws = torch.zeros((rows, 1024), dtype=torch.int32, device=DEV)
        idx.idx_paged_mqa_logits_decode_mxfp4(dev(q8), dev(w), g, 64, dev(pool.block_table), dev(ctx), out,
                                              sparse_idx=si, end=end, sbk=sbk, ws=ws)
        k = 256
        pos = torch.empty((rows, k), dtype=torch.int32, device=DEV)
        cols = torch.empty((rows, k), dtype=torch.int32, device=DEV)
        idx.idx_sparse_topk_remap(out, end, si, None, sbk, k, pos, col_scratch=cols, ws=ws)
        idx.idx_device_error()
        ref = O.sparse_logits_decode_mxfp4(q8, w, o, 64, pool.block_table, None, osi, oend, sbk)
        got = out.float().cpu().numpy()
        assert_logits_close(got, ref, f"sparse mxfp4 logits sbk {sbk}", bf16=True)
        c, p = cols.cpu().numpy(), pos.cpu().numpy()
        for r in range(rows):
            e = int(oend[r])
            assert_topk_values_exact(c[r], got[r, :e], k, f"row {r} sparse selection on its own scores")
            assert_topk_row(c[r], ref[r, :e], k, f"row {r} sparse selection vs oracle", bf16=True)
            m = min(k, e)
            assert np.array_equal(p[r, :m], O.sparse_remap_columns(c[r, :m], osi[r], 0, sbk))
            assert np.all(p[r, m:] == -1)


def test_mxfp4_decode_many_tiles_per_cta():
    # more tiles than two CTAs per SM can take at once: every CTA walks several
    # requests, their ragged tails and the look-ahead of the scale writes across
    # request boundaries; every row checked against the oracle
    rng = np.random.default_rng(98)
    ctx = rng.integers(1, 40000, 48).astype(np.int32)
    ctx[:4] = [1, 127, 128, 129]
    pool = W.make_pool(98, ctx)
    g, o = build_mx_caches(pool, 98)
    q8, w = W.make_q(99, len(ctx))
    out = torch.empty((len(ctx), int(ctx.max())), dtype=torch.float32, device=DEV)
    idx.idx_paged_mqa_logits_decode_mxfp4(dev(q8), dev(w), g, 64, dev(pool.block_table), dev(ctx), out)
    idx.idx_device_error()
    ref = O.paged_decode_logits_mxfp4(q8, w, o, 64, pool.block_table, ctx)
    got = out.cpu().numpy()
    for r in range(len(ctx)):
        L = int(ctx[r])
        assert_logits_close(got[r, :L], ref[r, :L], f"row {r}")


@pytest.mark.parametrize("next_n", [2, 3])
def test_mxfp4_hierarchical_mtp_rows_and_layer_reuse(next_n):
    # the V4.1 consumer layers on the MXFP4 cache with multi-token prediction:
    # next_n query rows per request (row r of request r // next_n sees
    # [0, L - next_n + j + 1)), one expansion reused by two layers, each layer's
    # scores, selection, positions and slots checked against the oracle
    from sparse_attention_indexer_fp8_gb300.pipeline import HierarchicalStep

    ctx = np.array([1000, 777, 4096, 2500, 64, 5], dtype=np.int32)
    B = len(ctx)
    rows = B * next_n
    pool = W.make_pool(400 + next_n, ctx)
    g, o = build_mx_caches(pool, 400 + next_n)
    cand = W.make_candidates(410 + next_n, rows, 16, 64, n_dup=3, n_pad=2, n_oob=2)
    r2r = np.repeat(np.arange(B), next_n).astype(np.int32)
    row_ke = np.array([O.decode_row_limit(int(ctx[r // next_n]), next_n, r % next_n) for r in range(rows)],
                      dtype=np.int32)
    k = 200
    st = HierarchicalStep(rows, cand.shape[1], 64, 64, k, 64, DEV, next_n=next_n, kv="mxfp4")
    st.expand(dev(cand), dev(ctx), dev(row_ke))
    osi, oend = O.expand_candidates(cand, None, row_ke, 64, 64)
    assert np.array_equal(st.sparse_idx.cpu().numpy(), osi) and np.array_equal(st.end.cpu().numpy(), oend)
    for layer in range(2):
        q8, w = W.make_q(420 + 10 * layer + next_n, rows)
        slots = st.score(dev(q8), dev(w), g, dev(pool.block_table), dev(ctx)).cpu().numpy()
        idx.idx_device_error()
        ref = O.sparse_logits_decode_mxfp4(q8, w, o, 64, pool.block_table, r2r, osi, oend, 64)
        got = st.logits.float().cpu().numpy()
        assert_logits_close(got, ref, f"layer {layer} sparse logits", bf16=True)
        cols, pos = st.cols.cpu().numpy(), st.positions.cpu().numpy()
        for r in range(rows):
            e = int(oend[r])
            assert_topk_values_exact(cols[r], got[r, :e], k, f"layer {layer} row {r}")
            assert_topk_row(cols[r], ref[r, :e], k, f"layer {layer} row {r} vs oracle", bf16=True)
            m = min(k, e)
            assert pos[r, :m].tolist() == [O.sparse_column_token(osi[r], int(c), 64) for c in cols[r, :m]]
            assert np.all(pos[r, m:] == -1)
        assert np.array_equal(slots, O.req_to_global_slots(pos, r2r, pool.block_table, 64, 64))


@pytest.mark.parametrize("block_size", [16, 64])
def test_mxfp4_gather_k_bitexact(block_size):
    # the prefill gather of every request: the codes and scale words the oracle reads
    ctx = np.array([300, 1, 65, 2049], dtype=np.int32)
    pool = W.make_pool(500 + block_size, ctx, block_size=block_size, extra_blocks=3)
    g, o = build_mx_caches(pool, 500 + block_size, block_size)
    for b in range(len(ctx)):
        n = int(ctx[b])
        codes = torch.full((n, 64), 0xAB, dtype=torch.uint8, device=DEV)
        scales = torch.full((n,), -1, dtype=torch.int32, device=DEV)
        idx.idx_gather_k_mxfp4(g, block_size, dev(pool.block_table[b]), n, codes, scales)
        idx.idx_device_error()
        opacked, oscales = O.mxfp4_gather_k(o, block_size, pool.block_table[b], n)
        assert np.array_equal(codes.cpu().numpy(), opacked), f"request {b} codes"
        assert np.array_equal(scales.cpu().numpy().view(np.uint8).reshape(n, 4), oscales), f"request {b} scales"


@pytest.mark.parametrize("sbk,out_bf16", [(16, True), (64, False)])
def test_mxfp4_sparse_prefill_logits_and_remap(sbk, out_bf16):
    # the V4.1 sparse prefill on the MXFP4 cache: gather one request's k, score the
    # candidate sparse blocks of rows that start at ks > 0, select and remap
    S, T = 3000, 40
    pool = W.make_pool(520, [S], extra_blocks=2)
    g, o = build_mx_caches(pool, 520)
    codes = torch.empty((S, 64), dtype=torch.uint8, device=DEV)
    scales = torch.empty((S,), dtype=torch.int32, device=DEV)
    idx.idx_gather_k_mxfp4(g, 64, dev(pool.block_table[0]), S, codes, scales)
    opacked, oscales = O.mxfp4_gather_k(o, 64, pool.block_table[0], S)
    q8, w = W.make_q(521, T)
    rng = np.random.default_rng(522)
    ks = (rng.integers(0, 60, T) * sbk).astype(np.int32)
    ke = np.minimum(ks + rng.integers(1, 2000, T), S).astype(np.int32)
    cand = W.make_candidates(523, T, 16, 40)
    R = 64 // sbk
    si = torch.empty((T, 16 * R), dtype=torch.int32, device=DEV)
    end = torch.empty(T, dtype=torch.int32, device=DEV)
    idx.idx_expand_candidates(dev(cand), dev(ks), dev(ke), 64, sbk, si, end)
    osi, oend = O.expand_candidates(cand, ks, ke, 64, sbk)
    assert np.array_equal(si.cpu().numpy(), osi) and np.array_equal(end.cpu().numpy(), oend)
    out = torch.empty((T, 16 * R * sbk), device=DEV, dtype=torch.bfloat16 if out_bf16 else torch.float32)
    ws = torch.zeros((T, 1024), dtype=torch.int32, device=DEV)
    idx.idx_mqa_logits_prefill_mxfp4(dev(q8), dev(w), codes, scales, out, si, end, sbk, ws=ws)
    ref = O.sparse_logits_prefill_mxfp4(q8, w, opacked, oscales, osi, oend, sbk)
    got = out.float().cpu().numpy()
    assert_logits_close(got, ref, "MXFP4 sparse prefill logits", bf16=out_bf16)
    k = 512
    pos = torch.empty((T, k), dtype=torch.int32, device=DEV)
    cols = torch.empty((T, k), dtype=torch.int32, device=DEV)
    idx.idx_sparse_topk_remap(out, end, si, dev(ks), sbk, k, pos, col_scratch=cols, ws=ws)
    idx.idx_device_error()
    assert not ws.any().item()
    pos, cols = pos.cpu().numpy(), cols.cpu().numpy()
    for r in range(T):
        e = int(oend[r])
        assert_topk_values_exact(cols[r], got[r, :e], k, f"row {r} on its own scores")
        assert_topk_row(cols[r], ref[r, :e], k, f"row {r} vs oracle", bf16=out_bf16)
        m = min(k, e)
        assert np.array_equal(pos[r, :m], O.sparse_remap_columns(cols[r, :m], osi[r], int(ks[r]), sbk))
        assert np.all(pos[r, m:] == -1)
