"""Pins for the oracle's MXFP4 indexer cache (CPU only).

The e2m1 / e8m0 codecs are checked against the OCP MX format table and
hand-worked rounding cases (golden fixture with its source), and the encoder
by brute force against every representable value; the quantiser against
hand-worked blocks, exact round trips and the saturation bound; the cache
layout against hand-computed byte offsets; the scoring against one-hot closed
forms, paging transparency and the sparse = dense-at-mapped-positions rule.
"""

import json
import os

import numpy as np
import pytest

from oracle import indexer as O
from oracle.codecs import E2M1_TABLE, bf16_decode, e2m1_decode, e2m1_encode, e4m3_decode, e8m0_decode
from sparse_attention_indexer_fp8_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _spec():
    with open(os.path.join(GOLDEN, "mxfp4.json")) as f:
        return json.load(f)


def test_e2m1_and_e8m0_golden_codes():
    spec = _spec()
    for code, value in spec["e2m1_codes"]:
        v = e2m1_decode(code)
        assert v == value and np.signbit(v) == np.signbit(value), (code, value)
    for x, code in spec["e2m1_rounding"]:
        assert e2m1_encode(x) == code, (x, code)
    for code, value in spec["e8m0_codes"]:
        assert e8m0_decode(code) == value
    assert np.isnan(e8m0_decode(255))


def test_e2m1_encode_is_nearest_with_ties_to_even_by_brute_force():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-8, 8, 20000), np.arange(-6.5, 6.75, 0.25),
                        rng.standard_normal(2000) * 1e-3])
    codes = e2m1_encode(x)
    vals = E2M1_TABLE[:8]                                # the eight magnitudes
    for xi, c in zip(x, codes):
        m = min(abs(xi), 6.0)
        d = np.abs(vals - m)
        best = np.nonzero(d == d.min())[0]
        mag_code = int(c) & 7
        assert mag_code in best, (xi, c)
        if len(best) == 2:                               # a tie: the code with the even mantissa bit
            assert mag_code % 2 == 0, (xi, c)
        assert (int(c) >> 3) == int(np.signbit(xi))
    # every representable value encodes to its own code
    assert np.array_equal(e2m1_encode(E2M1_TABLE), np.arange(16))


def test_mxfp4_quant_hand_worked_blocks():
    for blk in _spec()["blocks"]:
        k = np.zeros((1, 128), dtype=np.float32)
        j = 2                                            # third block of the token
        k[0, 32 * j:32 * j + 4] = blk["values"]
        codes, scales = O.mxfp4_quant(k)
        assert scales[0, j] == blk["scale_code"], blk["note"]
        assert list(codes[0, 32 * j:32 * j + 4]) == blk["codes"], blk["note"]
        assert np.all(codes[0, 32 * j + 4:32 * j + 32] == 0)
        # the other blocks are all zero: scale code 0, zero elements
        assert all(scales[0, i] == 0 for i in range(4) if i != j)


def test_mxfp4_quant_range_ends():
    k = np.zeros((3, 128), dtype=np.float32)
    k[0, :32] = np.float32(2.0 ** -130)                  # subnormal amax: exponent clamps to -127
    k[1, 32] = np.float32(1.5 * 2.0 ** 127)              # near the top: floor(log2) 127, shared 125
    k[1, 33] = np.float32(2.0 ** 126)
    k[2, 64:96] = np.float32(3.0 * 2.0 ** -20)
    codes, scales = O.mxfp4_quant(k)
    assert scales[0, 0] == 0 and np.all(codes[0, :32] == 0)          # 2^-130 / 2^-127 = 1/8 -> 0
    assert scales[1, 1] == 252 and codes[1, 32] == 0b0111 and codes[1, 33] == 0b0100   # 6 and 2 times 2^125
    assert scales[2, 2] == 127 - 21 and np.all(codes[2, 64:96] == 0b0111)   # 3 * 2^-20 = 6 * 2^-21


def test_mxfp4_round_trip_of_representable_tokens_and_error_bound():
    rng = np.random.default_rng(1)
    # tokens built from representable values whose block maximum is 4 or 6 times the scale
    n = 200
    codes = rng.integers(0, 16, (n, 128)).astype(np.uint8)
    codes[:, ::32] = rng.choice([6, 7, 14, 15], (n, 4))   # |max| in {4, 6}: floor(log2) - 2 = the scale
    sc = rng.integers(100, 150, (n, 4)).astype(np.uint8)
    vals = O.mxfp4_values(codes, sc).astype(np.float32)
    c2, s2 = O.mxfp4_quant(vals)
    assert np.array_equal(s2, sc)
    assert np.array_equal(e2m1_decode(c2), e2m1_decode(codes))     # -0 and +0 may differ in sign only
    # random tokens: each element within half a step of its block's grid, saturation within 2 scale units
    k = rng.standard_normal((500, 128)).astype(np.float32) * np.exp2(rng.integers(-8, 8, (500, 1)))
    c3, s3 = O.mxfp4_quant(k)
    deq = O.mxfp4_values(c3, s3)
    scale = np.repeat(e8m0_decode(s3), 32, axis=1)
    q = np.abs(k) / scale
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    err = np.abs(deq - k) / scale
    assert np.all(err <= np.where(q <= 6, step / 2, q - 6) + 1e-12)
    assert np.all(q < 8)                                  # floor(log2 amax) - 2 keeps every quotient below 8


def test_mxfp4_pack_and_cache_layout_hand_worked():
    assert list(O.mxfp4_pack(np.array([[1, 2, 3, 4] + [0] * 124]))[0, :2]) == [0x21, 0x43]
    bs = 16
    stride = O.mxfp4_block_stride(bs)
    assert stride == 1536 and O.mxfp4_block_stride(64) == 4608 and O.MXFP4_TOKEN_BYTES == 68
    cache = np.zeros((3, stride), dtype=np.uint8)
    k = np.zeros((2, 128), dtype=np.float32)
    k[0, 1] = 6.0                                        # dim 1: high nibble of byte 0, code 7
    k[0, 127] = -0.5                                     # dim 127: last block, scale 2^(floor(log2 .5)-2) = 2^-3
    k[1, 0] = 1.0
    O.mxfp4_k_quant_and_cache(k, [37, -1], cache, bs)    # slot 37 -> block 2, offset 5
    assert cache[2, 5 * 64] == 0x70                      # dim 0 = 0 (low nibble), dim 1 = code 7
    assert cache[2, 5 * 64 + 63] == 0xE0                 # dim 127 = -0.5 / 2^-3 = -4: code 14, high nibble
    assert list(cache[2, bs * 64 + 20:bs * 64 + 24]) == [127, 0, 0, 124]
    assert np.count_nonzero(cache) == 2 + 2
    c, s = O.mxfp4_cache_token(cache, bs, 2, 5)
    assert c[1] == 7 and c[127] == 0xE and list(s) == [127, 0, 0, 124]


def test_mxfp4_logits_one_hot_closed_form():
    rng = np.random.default_rng(2)
    for _ in range(20):
        h, d = int(rng.integers(0, 64)), int(rng.integers(0, 128))
        a = int(rng.integers(1, 126))
        kc = int(rng.integers(1, 16))
        e = int(rng.integers(110, 140))
        q8 = np.zeros((64, 128), dtype=np.uint8)
        q8[h, d] = a
        w = rng.standard_normal(64)
        codes = np.zeros((2, 128), dtype=np.uint8)
        scales = np.full((2, 4), 127, dtype=np.uint8)
        codes[0, d] = kc
        scales[0, d // 32] = e
        codes[1, (d + 32) % 128] = kc                    # another dim: contributes nothing
        out = O.logits_row_values(q8, w, O.mxfp4_values(codes, scales))
        assert out[0] == pytest.approx(w[h] * e4m3_decode(a) * e2m1_decode(kc) * 2.0 ** (e - 127), rel=1e-15, abs=0)
        assert out[1] == 0.0


def _mx_pool(seed, ctx, bs=64):
    pool = W.make_pool(seed, ctx)
    cache = np.zeros((pool.num_blocks, O.mxfp4_block_stride(bs)), dtype=np.uint8)
    ks = []
    for b in range(len(ctx)):
        kf = bf16_decode(W.make_k(seed, b, int(ctx[b])))
        O.mxfp4_k_quant_and_cache(kf, pool.slot_mapping(b), cache, bs)
        ks.append(kf)
    return pool, cache, ks


def test_mxfp4_paged_decode_equals_direct_scoring():
    # paging transparency: scores read through the shuffled block table equal scores of the
    # directly quantised contiguous k; the causal tail of MTP rows is -inf
    ctx = np.array([300, 129, 64])
    pool, cache, ks = _mx_pool(5, ctx)
    q8, w = W.make_q(5, 6)
    out = O.paged_decode_logits_mxfp4(q8, w, cache, 64, pool.block_table, ctx, next_n=2)
    for b in range(3):
        c, s = O.mxfp4_quant(ks[b])
        kv = O.mxfp4_values(c, s)
        for j in range(2):
            r = 2 * b + j
            lim = int(ctx[b]) - 2 + j + 1
            assert np.array_equal(out[r, :lim], O.logits_row_values(q8[r], w[r], kv[:lim]))
            assert np.all(np.isneginf(out[r, lim:ctx[b]])) and np.all(np.isnan(out[r, ctx[b]:]))


def test_mxfp4_scores_track_the_unquantised_scores():
    # sanity of the whole chain: MXFP4 k changes each score by at most the sum of the
    # per-element quantisation errors weighted by |w| |q|
    ctx = np.array([500])
    pool, cache, ks = _mx_pool(6, ctx)
    q8, w = W.make_q(6, 1)
    got = O.paged_decode_logits_mxfp4(q8, w, cache, 64, pool.block_table, ctx)[0]
    exact = O.logits_row_values(q8[0], w[0], ks[0].astype(np.float64))
    c, s = O.mxfp4_quant(ks[0])
    kerr = np.abs(O.mxfp4_values(c, s) - ks[0])
    bound = (np.abs(w[0])[:, None] * np.abs(e4m3_decode(q8[0]))).sum(0) @ kerr.T
    assert np.all(np.abs(got - exact) <= bound * (1 + 1e-12) + 1e-12)


def test_mxfp4_sparse_logits_equal_dense_at_mapped_positions():
    ctx = np.array([1000, 777, 2048])
    pool, cache, _ = _mx_pool(7, ctx)
    q8, w = W.make_q(7, 3)
    cand = W.make_candidates(7, 3, 8, 16, n_dup=2, n_pad=1, n_oob=1)
    dense = O.paged_decode_logits_mxfp4(q8, w, cache, 64, pool.block_table, ctx)
    for sbk, cbs in ((64, 64), (16, 64)):
        si, end = O.expand_candidates(cand, None, ctx, cbs, sbk)
        sp = O.sparse_logits_decode_mxfp4(q8, w, cache, 64, pool.block_table, None, si, end, sbk)
        for r in range(3):
            for c in range(sp.shape[1]):
                if c < end[r]:
                    assert sp[r, c] == dense[r, O.sparse_column_token(si[r], c, sbk)]
                else:
                    assert sp[r, c] == -np.inf


def test_mxfp4_gather_equals_token_by_token_reads():
    ctx = np.array([300, 129])
    pool, cache, _ = _mx_pool(8, ctx, bs=64)
    for b in range(2):
        pos = np.random.default_rng(b).permutation(int(ctx[b]))[:50]
        got = O.mxfp4_gather_values(cache, 64, pool.block_table[b], pos)
        for i, p in enumerate(pos):
            c, s = O.mxfp4_cache_token(cache, 64, int(pool.block_table[b][p // 64]), int(p) % 64)
            assert np.array_equal(got[i], O.mxfp4_values(c, s)[0])


def test_mxfp4_gather_k_equals_cache_reads_and_quantised_k():
    # the prefill gather of one request: row p holds token p's packed codes and
    # scale codes; decoded, the rows equal both the vectorised paged read and the
    # MXFP4 conversion of the k that filled the cache
    ctx = np.array([300, 129])
    pool, cache, ks = _mx_pool(9, ctx, bs=64)
    for b in range(2):
        n = int(ctx[b])
        packed, scales = O.mxfp4_gather_k(cache, 64, pool.block_table[b], n)
        assert packed.shape == (n, 64) and scales.shape == (n, 4)
        for p in (0, 1, 63, 64, n - 1):
            c, s = O.mxfp4_cache_token(cache, 64, int(pool.block_table[b][p // 64]), p % 64)
            assert np.array_equal(O.mxfp4_unpack(packed[p:p + 1])[0], c) and np.array_equal(scales[p], s)
        vals = O.mxfp4_values(O.mxfp4_unpack(packed), scales)
        assert np.array_equal(vals, O.mxfp4_gather_values(cache, 64, pool.block_table[b], range(n)))
        assert np.array_equal(vals, O.mxfp4_values(*O.mxfp4_quant(ks[b])))


def test_mxfp4_sparse_logits_prefill_one_hot_closed_form():
    rng = np.random.default_rng(10)
    S, T, sbk = 256, 3, 16
    for _ in range(10):
        h, d, t = int(rng.integers(0, 64)), int(rng.integers(0, 128)), int(rng.integers(0, S))
        a, kc, e = int(rng.integers(1, 126)), int(rng.integers(1, 16)), int(rng.integers(110, 140))
        q8 = np.zeros((T, 64, 128), dtype=np.uint8)
        q8[:, h, d] = a
        w = rng.standard_normal((T, 64))
        codes = np.zeros((S, 128), dtype=np.uint8)
        scales = np.full((S, 4), 127, dtype=np.uint8)
        codes[t, d] = kc
        scales[t, d // 32] = e
        packed = O.mxfp4_pack(codes)
        si = np.tile(np.arange(S // sbk), (T, 1))
        end = np.array([S, t + 1, t])                      # the last row stops just before token t
        out = O.sparse_logits_prefill_mxfp4(q8, w, packed, scales, si, end, sbk)
        for r in range(T):
            want = np.zeros(S)
            want[t] = w[r, h] * e4m3_decode(a) * e2m1_decode(kc) * 2.0 ** (e - 127)
            e_r = int(end[r])
            assert np.allclose(out[r, :e_r], want[:e_r], rtol=1e-15, atol=0)
            assert np.all(np.isneginf(out[r, e_r:]))


def test_mxfp4_sparse_logits_prefill_equal_dense_at_mapped_positions():
    # rows of a prefill chunk whose requests start at ks > 0: every valid sparse
    # column equals the logit of its absolute token over the whole quantised k
    rng = np.random.default_rng(11)
    S, T = 700, 6
    k = rng.standard_normal((S, 128)).astype(np.float32)
    codes, scales = O.mxfp4_quant(k)
    packed = O.mxfp4_pack(codes)
    kv = O.mxfp4_values(codes, scales)
    q8, w = W.make_q(11, T)
    for sbk, cbs in ((64, 64), (16, 64), (8, 32)):
        row_ks = np.array([0, sbk, 3 * sbk, 128, 2 * sbk, 5 * sbk])
        row_ke = np.array([700, 650, 400, 300, 2 * sbk + 1, 700])
        cand = rng.integers(-1, 12, (T, 8))
        si, end = O.expand_candidates(cand, row_ks, row_ke, cbs, sbk)
        sp = O.sparse_logits_prefill_mxfp4(q8, w, packed, scales, si, end, sbk)
        assert np.count_nonzero(end) >= T // 2
        for r in range(T):
            full = O.logits_row_values(q8[r], w[r], kv)
            for c in range(sp.shape[1]):
                if c < end[r]:
                    tok = O.sparse_column_token(si[r], c, sbk)
                    assert row_ks[r] <= tok < row_ke[r]
                    assert sp[r, c] == full[tok]
                else:
                    assert sp[r, c] == -np.inf
