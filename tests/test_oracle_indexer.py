"""Pins for the oracle's indexer functions (CPU only).

Each function is checked against something other than itself: hand-worked
examples (golden fixtures with their source), closed forms with one-hot inputs,
exact rational arithmetic, brute force over all subsets, token-level brute
force, invariants (linearity, paging transparency, sparse = dense-masked), and
library routines on special cases.
"""

import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import indexer as O
from oracle.codecs import bf16_decode, bf16_encode, e4m3_decode, e4m3_encode
from sparse_attention_indexer_fp8_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- k quant

def test_k_quant_hand_worked():
    k = np.zeros((4, 128), dtype=np.float32)
    k[0, 5] = 448.0                      # scale exactly 1: the byte is the e4m3 max
    k[2, 0] = 7.0                        # amax 7 -> scale 7/448 = 2^-6 exactly
    k[2, 1] = 0.5                        # 0.5 / 2^-6 = 32 -> 0x60
    k[2, 2] = -3.5                       # -224 -> 0xF6
    k[2, 3] = 2.0 ** -16                 # 2^-10 after scaling: tie with 0 -> +0
    k[3, :] = -1.0                       # amax 1: every value maps to -448 (or just below)
    k8, s = O.k_quant(k)
    assert s[0] == np.float32(1.0)
    assert k8[0, 5] == 0x7E and np.count_nonzero(k8[0]) == 1
    assert s[1] == 0 and not k8[1].any()
    assert s[2] == np.float32(2.0 ** -6)
    assert list(k8[2, :4]) == [0x7E, 0x60, 0xF6, 0x00]
    assert s[3] == np.float32(1.0) / np.float32(448.0)
    assert np.all(k8[3] == 0xFE)


def test_k_quant_matches_torch_cast():
    # the division and the cast done by library routines for a random batch
    rng = np.random.default_rng(3)
    k = (rng.standard_normal((64, 128)) * rng.uniform(0.01, 100, (64, 1))).astype(np.float32)
    k8, s = O.k_quant(k)
    kt = torch.from_numpy(k)
    st = kt.abs().amax(dim=1) / torch.tensor(448.0)
    assert np.array_equal(st.numpy(), s)
    ref = (kt / st[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref, k8)


def test_k_quant_bf16_inputs_and_underflow():
    kb = W.make_k(5, 0, 16)
    k = bf16_decode(kb)
    k8, s = O.k_quant(k)
    assert np.all(s > 0)
    recon = e4m3_decode(k8) * s[:, None]
    assert np.all(np.abs(recon - k) <= np.abs(k) * 2.0 ** -4 + s[:, None] * 2.0 ** -9 + 1e-30)
    tiny = np.zeros((1, 128), dtype=np.float32)
    tiny[0, 0] = np.float32(1e-45)       # smallest subnormal: amax/448 underflows to 0
    k8, s = O.k_quant(tiny)
    assert s[0] == 0 and not k8.any()


def test_ue8m0_scales_hand_worked_and_bounds():
    # amax 448 -> 1 (already a power of two); 500 -> 500/448 = 1.116 -> 2;
    # 224 -> 0.5; 300 -> 0.6696 -> 1; 0 -> 0 (zero bytes)
    k = np.zeros((5, 128), dtype=np.float32)
    for i, a in enumerate([448.0, 500.0, 224.0, 300.0, 0.0]):
        k[i, 7] = a
        k[i, 8] = -a / 2
    k8, s = O.k_quant(k, ue8m0=True)
    assert s.tolist() == [1.0, 2.0, 0.5, 1.0, 0.0]
    assert e4m3_decode(k8[1, 7:9]).tolist() == [256.0, -128.0]      # 500/2 = 250 -> 256 (RNE), -125 -> -128
    assert e4m3_decode(k8[3, 7:9]).tolist() == [288.0, -144.0]      # 300, -150 rounded to e4m3
    assert not k8[4].any()
    # random rows: a power of two in [amax/448, 2 amax/448), every code within range
    rng = np.random.default_rng(30)
    kr = (rng.standard_normal((200, 128)) * rng.uniform(1e-3, 1e3, (200, 1))).astype(np.float32)
    k8, s = O.k_quant(kr, ue8m0=True)
    base = (np.max(np.abs(kr), axis=1) / np.float32(448)).astype(np.float32)
    m, _ = np.frexp(s.astype(np.float64))
    assert np.all(m == 0.5) and np.all(s >= base) and np.all(s < 2 * base)
    # the division by a power of two is exact: codes are the fp32 scaling's codes
    assert np.array_equal(k8, e4m3_encode(kr.astype(np.float64) / s[:, None]))


def test_cache_layout_hand_worked():
    bs, stride = 64, W.block_stride_bytes(64)
    assert stride == 8704
    cache = np.zeros((4, stride), dtype=np.uint8)
    k = np.zeros((2, 128), dtype=np.float32)
    k[0, 0] = 448.0
    k[1, 127] = -448.0
    O.k_quant_and_cache(k, [130, -1], cache, bs)       # slot 130 -> block 2, offset 2
    assert cache[2, 256] == 0x7E                        # value row at offset 2*128
    assert np.count_nonzero(cache) == 1 + 2             # value byte + scale 1.0 = 0x3F800000
    assert list(cache[2, 8192 + 8:8192 + 12]) == [0x00, 0x00, 0x80, 0x3F]
    k8, s = O.cache_token(cache, bs, 2, 2)
    assert k8[0] == 0x7E and s == 1.0


# ---------------------------------------------------------------- logits

def _one_hot_q(rows, h, d, code):
    q8 = np.zeros((rows, 64, 128), dtype=np.uint8)
    q8[:, h, d] = code
    return q8


def test_logits_one_hot_closed_form():
    rng = np.random.default_rng(0)
    for _ in range(20):
        h, d, d2 = rng.integers(0, 64), rng.integers(0, 128), rng.integers(0, 128)
        a, b = int(rng.integers(1, 126)), int(rng.integers(1, 126))
        q8 = _one_hot_q(1, h, d, a)
        w = rng.standard_normal((1, 64))
        k8 = np.zeros((3, 128), dtype=np.uint8)
        k8[0, d] = b
        k8[1, d2] = b                                     # other dim: contributes only if d2 == d
        kscale = np.array([0.5, 2.0, 3.0], dtype=np.float32)
        out = O.logits_row(q8[0], w[0], k8, kscale)
        expect0 = w[0, h] * e4m3_decode(a) * e4m3_decode(b) * 0.5
        expect1 = w[0, h] * e4m3_decode(a) * e4m3_decode(b) * 2.0 if d2 == d else 0.0
        assert out[0] == pytest.approx(expect0, rel=1e-15, abs=0)
        assert out[1] == pytest.approx(expect1, rel=1e-15, abs=1e-300)
        assert out[2] == 0.0


def test_logits_head_dot_is_exact():
    # the per-head dot product is exact in fp64; compare with rational arithmetic
    rng = np.random.default_rng(1)
    q8 = rng.integers(0, 254, (64, 128)).astype(np.uint8)
    q8[q8 == 0x7F] = 0x7E
    k8 = rng.integers(0, 254, (2, 128)).astype(np.uint8)
    k8[k8 == 0x7F] = 0x7E
    w = np.zeros(64)
    for h in (0, 17, 63):
        w[:] = 0
        w[h] = 1.0
        got = O.logits_row(q8, w, k8, np.ones(2, dtype=np.float32))
        for s in range(2):
            exact = sum(Fraction(float(e4m3_decode(q8[h, d]))) * Fraction(float(e4m3_decode(k8[s, d])))
                        for d in range(128))
            assert Fraction(got[s]) == exact


def test_logits_linear_in_weights_and_scale():
    rng = np.random.default_rng(2)
    q8, w = W.make_q(9, 2)
    w = w.astype(np.float64)
    k8, ks = W.make_random_cache_tokens(9, 50)
    a = O.logits_row(q8[0], w[0], k8, ks)
    b = O.logits_row(q8[0], w[1], k8, ks)
    c = O.logits_row(q8[0], w[0] + w[1], k8, ks)
    assert np.allclose(a + b, c, rtol=1e-12, atol=1e-18)
    ks2 = ks.copy()
    ks2[7] *= 2
    d = O.logits_row(q8[0], w[0], k8, ks2)
    assert d[7] == pytest.approx(2 * a[7], rel=1e-14)
    assert np.array_equal(np.delete(d, 7), np.delete(a, 7))
    # heads are interchangeable: permuting q heads together with the weights changes nothing
    perm = rng.permutation(64)
    e = O.logits_row(q8[0][perm], w[0][perm], k8, ks)
    assert np.allclose(e, a, rtol=1e-12, atol=1e-18)


def test_prefill_logits_masks_outside_row_limits():
    q8, w = W.make_q(4, 3)
    k8, ks = W.make_random_cache_tokens(4, 40)
    out = O.mqa_logits(q8, w, k8, ks, [0, 5, 10], [40, 6, 10])
    assert np.all(np.isfinite(out[0]))
    assert np.isfinite(out[1, 5]) and np.sum(np.isfinite(out[1])) == 1
    assert not np.isfinite(out[2]).any()
    assert np.all(out[1, :5] == -np.inf)


def test_paged_decode_equals_contiguous_scoring():
    """Paging is transparent: scores read through a shuffled block table equal the gathered ones."""
    wl = W.tiny_decode()
    pool = wl.pool
    cache = np.zeros((pool.num_blocks, W.block_stride_bytes()), dtype=np.uint8)
    per_req = []
    for b in range(wl.batch):
        kb = bf16_decode(W.make_k(wl.seed, b, int(pool.ctx_lens[b])))
        O.k_quant_and_cache(kb, pool.slot_mapping(b), cache, pool.block_size)
        per_req.append(O.k_quant(kb))
    paged = O.paged_decode_logits(wl.q8, wl.w, cache, pool.block_size, pool.block_table, pool.ctx_lens, 1)
    for b in range(wl.batch):
        L = int(pool.ctx_lens[b])
        k8, ks = per_req[b]
        ref = O.logits_row(wl.q8[b], wl.w[b], k8, ks)
        assert np.array_equal(paged[b, :L], ref)
        assert np.all(np.isnan(paged[b, L:]))
    # next_n = 2: the first query of each request cannot see the second one's token
    q8 = np.repeat(wl.q8, 2, axis=0)
    w = np.repeat(wl.w, 2, axis=0)
    p2 = O.paged_decode_logits(q8, w, cache, pool.block_size, pool.block_table, pool.ctx_lens, 2)
    for b in range(wl.batch):
        L = int(pool.ctx_lens[b])
        assert p2[2 * b, L - 1] == -np.inf and np.isfinite(p2[2 * b, L - 2])
        assert np.isfinite(p2[2 * b + 1, L - 1])


def test_gather_roundtrip():
    bs = 16
    stride = W.block_stride_bytes(bs)
    k = bf16_decode(W.make_k(3, 0, 100))
    table = np.array([5, 0, 3, 7, 1, 2, 6])
    cache = np.zeros((8, stride), dtype=np.uint8)
    slots = table[np.arange(100) // bs] * bs + np.arange(100) % bs
    O.k_quant_and_cache(k, slots, cache, bs)
    k8, ks = O.gather_k(cache, bs, table, 100)
    k8r, ksr = O.k_quant(k)
    assert np.array_equal(k8, k8r) and np.array_equal(ks, ksr)


# ---------------------------------------------------------------- top-k

def _brute_force_topk_sets(vals, k):
    """Every k-subset whose minimum is at least the maximum of the rest (all valid answers)."""
    n = len(vals)
    good = []
    for comb in itertools.combinations(range(n), k):
        rest = [vals[i] for i in range(n) if i not in comb]
        if not rest or min(vals[i] for i in comb) >= max(rest):
            good.append(set(comb))
    return good


def test_topk_brute_force_small():
    rng = np.random.default_rng(5)
    for trial in range(200):
        n = int(rng.integers(1, 12))
        k = int(rng.integers(1, 6))
        vals = rng.integers(-3, 4, n).astype(np.float64)   # many ties
        ks = int(rng.integers(0, 3))
        row = np.concatenate([np.full(ks, 99.0), vals])    # columns before ks must be ignored
        got = O.topk_row(row, ks, ks + n, k)
        if n <= k:
            assert list(got[:n]) == list(range(n)) and np.all(got[n:] == -1)
            continue
        sel = set(int(i) for i in got)
        valid = _brute_force_topk_sets(list(vals), k)
        assert sel in valid
        # tie rule: the lexicographically smallest valid set (lower index wins)
        assert sorted(sel) == min(sorted(s) for s in valid)


# ------------------------------------------------- q preparation (RoPE + quant)

def _cos_sin_table(max_pos, base=10000.0):
    i = np.arange(32, dtype=np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * base ** (-2.0 * i / 64.0)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def test_q_rope_hand_worked():
    # one head: x_0 = 2, x_32 = 4 (a NeoX pair), c = 0.5, s = 0.75 (exact in binary):
    # y_0 = 2*0.5 - 4*0.75 = -2, y_32 = 4*0.5 + 2*0.75 = 3.5 (both e4m3 values at
    # scale 1); dim 100 passes through. Then 4.25 (x_1 = x_33 = ...) checks rounding:
    # x_1 = 3, x_33 = 4 give y_33 = 4*0.5 + 3*0.75 = 4.25, which e4m3 rounds (tie, even) to 4.
    q = np.zeros((1, 64, 128), dtype=np.float32)
    q[0, 0, 0], q[0, 0, 32], q[0, 0, 100] = 2.0, 4.0, 448.0
    q[0, 0, 1], q[0, 0, 33] = 3.0, 4.0
    cs = np.zeros((1, 64), dtype=np.float32)
    cs[0, :32], cs[0, 32:] = 0.5, 0.75
    w = np.full((1, 64), 2.0, dtype=np.float32)
    q8, w_out, scale = O.q_rope_quant(q, [0], cs, w, 0.5, 0.25)
    assert scale[0, 0] == 1.0                      # amax 448 -> scale 1
    dec = e4m3_decode(q8[0, 0])
    assert dec[0] == -2.0 and dec[32] == 3.5 and dec[100] == 448.0
    assert dec[1] == -1.5 and dec[33] == 4.0 and not dec[[2, 34, 64]].any()
    assert w_out[0, 0] == 2.0 * 1.0 * 0.5 * 0.25   # weights absorb scale * softmax * n_head
    assert np.all(scale[0, 1:] == 0) and np.all(q8[0, 1:] == 0) and np.all(w_out[0, 1:] == 0)


def test_q_rope_quarter_turns_are_exact():
    # c = 0, s = 1: (x_a, x_b) -> (-x_b, x_a); c = -1, s = 0: negation; identity for c = 1, s = 0
    rng = np.random.default_rng(21)
    q = rng.standard_normal((4, 64, 128)).astype(np.float32)
    w = rng.standard_normal((4, 64)).astype(np.float32)
    for interleaved in (False, True):
        a, b = O.rope_pairs(interleaved)
        for c_val, s_val in [(0.0, 1.0), (-1.0, 0.0), (1.0, 0.0)]:
            cs = np.zeros((1, 64), dtype=np.float32)
            cs[0, :32], cs[0, 32:] = c_val, s_val
            q8, w_out, scale = O.q_rope_quant(q, np.zeros(4, int), cs, w, 1.0, 1.0, interleaved)
            y = q.copy()
            y[:, :, a] = c_val * q[:, :, a] - s_val * q[:, :, b]
            y[:, :, b] = c_val * q[:, :, b] + s_val * q[:, :, a]
            k8, ks = O.k_quant(y.reshape(-1, 128))          # the pinned per-128 quantiser
            assert np.array_equal(q8.reshape(-1, 128), k8) and np.array_equal(scale.reshape(-1), ks)
            assert np.array_equal(w_out, w * ks.reshape(4, 64))


def test_q_rope_preserves_pair_norms_and_styles_agree():
    rng = np.random.default_rng(22)
    q = rng.standard_normal((6, 64, 128)).astype(np.float32)
    cs = _cos_sin_table(4096)
    pos = rng.integers(0, 4096, 6)
    w = np.ones((6, 64), dtype=np.float32)
    # rotation of each pair keeps its length (fp32 rounding only)
    for interleaved in (False, True):
        a, b = O.rope_pairs(interleaved)
        q8, _, scale = O.q_rope_quant(q, pos, cs, w, 1.0, 1.0, interleaved)
        y = e4m3_decode(q8).astype(np.float64) * scale[:, :, None]
        n_in = np.hypot(q[:, :, a], q[:, :, b])
        n_out = np.hypot(y[:, :, a], y[:, :, b])
        assert np.allclose(n_in, n_out, rtol=0.07, atol=0.07 * scale[:, :, None])   # e4m3 error
    # the interleaved pairing is the NeoX pairing applied to permuted dims
    perm = np.concatenate([np.arange(0, 64, 2), np.arange(1, 64, 2), np.arange(64, 128)])
    q8_i, w_i, _ = O.q_rope_quant(q, pos, cs, w, 1.0, 1.0, True)
    q8_n, w_n, _ = O.q_rope_quant(q[:, :, perm], pos, cs, w, 1.0, 1.0, False)
    assert np.array_equal(q8_i[:, :, perm], q8_n) and np.array_equal(w_i, w_n)


def test_q_rope_quant_folded_weights_reproduce_the_unfolded_score():
    # [DSA] step ④: with every coefficient in the weights, the scoring formula on
    # (q8, w_out) equals sum_h w * softmax_scale * n_head_scale * (rope(q)_h . k)
    # up to the e4m3 rounding of q
    rng = np.random.default_rng(23)
    q = rng.standard_normal((3, 64, 128)).astype(np.float32)
    w = (rng.standard_normal((3, 64)) / 8).astype(np.float32)
    cs = _cos_sin_table(64)
    pos = np.array([0, 17, 63])
    ss, nhs = 128 ** -0.5, 64 ** -0.5
    q8, w_out, scale = O.q_rope_quant(q, pos, cs, w, ss, nhs)
    k = rng.standard_normal((50, 128)).astype(np.float32)
    k8, ks = O.k_quant(k)
    a, b = O.rope_pairs(False)
    for t in range(3):
        c, s = cs[pos[t], :32].astype(np.float64), cs[pos[t], 32:].astype(np.float64)
        y = q[t].astype(np.float64)
        ya, yb = y[:, a] * c - y[:, b] * s, y[:, b] * c + y[:, a] * s
        y[:, a], y[:, b] = ya, yb
        kd = e4m3_decode(k8).astype(np.float64) * ks[:, None]
        exact = (w[t].astype(np.float64) * ss * nhs) @ (y @ kd.T)
        got = O.logits_row(q8[t], w_out[t], k8, ks)
        err_bound = (np.abs(w[t].astype(np.float64) * ss * nhs) @ np.abs(y @ kd.T)) * 2.0 ** -4 + 1e-9
        assert np.all(np.abs(got - exact) <= err_bound)


def test_q_rope_bf16_weights_are_the_fp32_result_rounded_once():
    # "V4.1 索引器接入稀疏 MQA logits", 实现拆解 item 5 / test list: bf16 weights equal the
    # fp32 weights rounded once; the rounding is checked against PyTorch's cast
    rng = np.random.default_rng(24)
    q = rng.standard_normal((5, 64, 128)).astype(np.float32)
    w = rng.standard_normal((5, 64)).astype(np.float32)
    _, w_out, _ = O.q_rope_quant(q, np.zeros(5, int), _cos_sin_table(1), w, 128 ** -0.5, 64 ** -0.5)
    ref = torch.from_numpy(w_out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_encode(w_out), ref)


def test_q_rope_out_of_range_position_zeroes_the_token():
    q = np.ones((2, 64, 128), dtype=np.float32)
    w = -np.ones((2, 64), dtype=np.float32)
    q8, w_out, scale = O.q_rope_quant(q, [0, 5], _cos_sin_table(3), w, 1.0, 1.0)
    assert np.all(q8[1] == 0) and np.all(scale[1] == 0) and np.all(w_out[1] == 0)
    assert np.all(scale[0] > 0)


# ------------------------------------------------- context-parallel merge

def test_dcp_merge_hand_worked():
    # shard 0 holds positions 0..9, shard 1 positions 10..; three candidates each.
    # Sorted by value then position: 5@2, 4@11, 3@0, 3@15, 1@7; the empty one is dropped.
    vals = np.array([5.0, 3.0, 1.0, 4.0, 3.0, -np.inf])
    idx = np.array([2, 0, 7, 1, 5, -1])
    pos, v = O.dcp_topk_merge_row(vals, idx, [0, 10], 3, 4)
    assert pos.tolist() == [2, 11, 0, 15] and v.tolist() == [5.0, 4.0, 3.0, 3.0]
    pos, v = O.dcp_topk_merge_row(vals, idx, [0, 10], 3, 7)
    assert pos.tolist() == [2, 11, 0, 15, 7, -1, -1]
    assert v[:5].tolist() == [5.0, 4.0, 3.0, 3.0, 1.0] and np.all(np.isneginf(v[5:]))
    # indices already global: no offsets
    pos, _ = O.dcp_topk_merge_row(vals, np.array([2, 0, 7, 11, 15, -1]), None, 3, 4)
    assert pos.tolist() == [2, 11, 0, 15]


def _shard_bounds(rng, n, n_shards):
    cuts = np.sort(rng.integers(0, n + 1, n_shards - 1))
    return np.concatenate([[0], cuts, [n]]).astype(np.int64)


def test_dcp_merge_of_local_topk_equals_global_topk():
    # The exactness claim of the context-parallel merge: every member of the
    # global top-k is in the local top-k of its own shard, so merging the local
    # lists reproduces the whole-row selection (same tie rule: lower position).
    rng = np.random.default_rng(11)
    for trial in range(300):
        n = int(rng.integers(1, 60))
        k = int(rng.integers(1, 12))
        n_shards = int(rng.integers(1, 6))
        row = rng.integers(-4, 5, n).astype(np.float64) if trial % 2 else rng.standard_normal(n)
        b = _shard_bounds(rng, n, n_shards)
        cv = np.full(n_shards * k, -np.inf)
        ci = np.full(n_shards * k, -1, dtype=np.int64)
        for s in range(n_shards):
            loc = O.topk_row(row, int(b[s]), int(b[s + 1]), k)
            ci[s * k:(s + 1) * k] = loc
            ok = loc >= 0
            cv[s * k:(s + 1) * k][ok] = row[b[s] + loc[ok]]
        pos, v = O.dcp_topk_merge_row(cv, ci, b[:-1], k, k)
        ref = O.topk_row(row, 0, n, k)
        m = min(n, k)
        assert sorted(pos[:m].tolist()) == sorted(ref[:m].tolist()) and np.all(pos[m:] == -1)
        assert np.array_equal(v[:m], row[pos[:m]]) and np.all(np.diff(v[:m]) <= 0)


def test_dcp_merge_interleaved_shards_equal_global_topk():
    # tokens dealt round-robin: shard s holds positions s, s + S, s + 2S, ...;
    # local index j of shard s is global position s + j * S
    rng = np.random.default_rng(13)
    pos, _ = O.dcp_topk_merge_row([3.0, 1.0, 2.0, -np.inf], [1, 0, 0, -1], [0, 1], 2, 3, 2)
    assert pos.tolist() == [2, 1, 0]                       # 3@(0+1*2), 2@(1+0*2), 1@(0+0*2)
    for trial in range(200):
        n = int(rng.integers(1, 50))
        k = int(rng.integers(1, 10))
        S = int(rng.integers(1, 5))
        row = rng.integers(-3, 4, n).astype(np.float64)
        cv = np.full(S * k, -np.inf)
        ci = np.full(S * k, -1, dtype=np.int64)
        for s in range(S):
            loc_row = row[s::S]
            loc = O.topk_row(loc_row, 0, len(loc_row), k)
            ci[s * k:(s + 1) * k] = loc
            ok = loc >= 0
            cv[s * k:(s + 1) * k][ok] = loc_row[loc[ok]]
        got, _ = O.dcp_topk_merge(cv[None], ci[None], np.arange(S)[None], k, k, S)
        m = min(n, k)
        assert sorted(got[0, :m].tolist()) == sorted(O.topk_row(row, 0, n, k)[:m].tolist())


def test_dcp_merge_brute_force_small():
    # any candidate multiset: the merged set is one of the maximal k-subsets
    rng = np.random.default_rng(12)
    for _ in range(200):
        k_local = int(rng.integers(1, 4))
        n_shards = int(rng.integers(1, 4))
        k = int(rng.integers(1, 6))
        n = n_shards * k_local
        vals = rng.integers(-2, 3, n).astype(np.float64)
        idx = rng.permutation(20)[:n]
        empty = rng.random(n) < 0.25
        idx[empty] = -1
        vals[empty] = -np.inf
        offs = np.arange(n_shards) * 100
        pos, v = O.dcp_topk_merge_row(vals, idx, offs, k_local, k)
        glob = [int(offs[j // k_local] + idx[j]) for j in range(n) if idx[j] >= 0]
        gval = [vals[j] for j in range(n) if idx[j] >= 0]
        m = min(len(glob), k)
        assert np.all(pos[m:] == -1) and np.all(np.isneginf(v[m:]))
        if m == len(glob):
            assert sorted(pos[:m].tolist()) == sorted(glob)
            continue
        chosen = {glob.index(int(p)) for p in pos[:m]}
        assert chosen in _brute_force_topk_sets(gval, k)


def test_topk_values_match_torch_topk():
    x = W.make_logits(8, 4, 5000)
    got = O.topk(x, None, [5000, 4000, 2048, 100], 2048)
    for r in range(4):
        n = [5000, 4000, 2048, 100][r]
        sel = got[r][got[r] >= 0]
        assert len(sel) == min(n, 2048) and len(set(sel.tolist())) == len(sel)
        ref = torch.topk(torch.from_numpy(x[r, :n]).double(), min(n, 2048)).values.numpy()
        assert np.array_equal(np.sort(x[r, sel].astype(np.float64)), np.sort(ref))


# ---------------------------------------------------------------- expansion

def test_expand_golden():
    with open(os.path.join(GOLDEN, "expand_candidates.json")) as f:
        spec = json.load(f)
    for c in spec["cases"]:
        si, end = O.expand_candidates_row(c["cand"], c["ks"], c["ke"], c["cand_block_size"], c["sbk"])
        assert list(si) == c["sparse_idx"], c["note"]
        assert end == c["end"], c["note"]


def test_expand_brute_force_invariants():
    rng = np.random.default_rng(6)
    for trial in range(400):
        sbk = int(rng.choice([8, 16, 64]))
        R = int(rng.choice([1, 2, 4]))
        cbs = sbk * R
        K = int(rng.choice([1, 2, 4, 8, 16]))
        ks = sbk * int(rng.integers(0, 4))
        ke = ks + int(rng.integers(0, 12 * cbs))
        nblk = (ke - ks + cbs - 1) // cbs + 2
        cand = rng.integers(-1, nblk + 1, K)
        si, end = O.expand_candidates_row(cand, ks, ke, cbs, sbk)
        # token-level brute force: relative position x is covered when its candidate block was published
        pub = set(int(c) for c in cand if c >= 0)
        covered = [x for x in range(ke - ks) if x // cbs in pub]
        assert end == len(covered)
        # the valid prefix lists the covered sparse blocks once each, ascending, anchored at ks // sbk
        blocks = sorted(set((ks + x) // sbk for x in covered))
        n = len(blocks)
        assert list(si[:n]) == blocks
        if n:
            assert np.all(si[n:] == blocks[-1])
        else:
            assert np.all(si == ks // sbk)
        # columns [0, end) address exactly the covered tokens
        toks = [O.sparse_column_token(si, c, sbk) for c in range(end)]
        assert toks == [ks + x for x in covered]


# ---------------------------------------------------------------- remap and slots

def test_slot_remap_golden():
    with open(os.path.join(GOLDEN, "slot_remap.json")) as f:
        spec = json.load(f)
    bt = np.array([spec["block_table"]])
    for c in spec["cases"]:
        out = O.req_to_global_slots(np.array([[c["local"]]]), None, bt, spec["block_size"], c["block_span"])
        assert out[0, 0] == c["slot"], c
    for c in spec["span_cases"]:
        if c["span"] is None:
            with pytest.raises(ValueError):
                O.packed_block_span(c["block_stride"], c["token_stride"])
        else:
            assert O.packed_block_span(c["block_stride"], c["token_stride"]) == c["span"]


def test_slots_span_equal_block_size_is_the_plain_slot():
    # with block_span == block_size the slot is the ordinary block*block_size + offset
    pool = W.make_pool(3, [300, 70])
    local = np.array([[0, 5, 299, -1], [69, 64, -1, -1]])
    out = O.req_to_global_slots(local, None, pool.block_table, 64, 64)
    for b in range(2):
        sm = pool.slot_mapping(b)
        for i in range(4):
            v = local[b, i]
            assert out[b, i] == (-1 if v < 0 else sm[v])


# ---------------------------------------------------------------- sparse path

def _tiny_hier():
    ctx = np.array([1000, 777, 2048], dtype=np.int32)
    pool = W.make_pool(21, ctx)
    cache = np.zeros((pool.num_blocks, W.block_stride_bytes()), dtype=np.uint8)
    for b in range(3):
        O.k_quant_and_cache(bf16_decode(W.make_k(21, b, int(ctx[b]))), pool.slot_mapping(b), cache, 64)
    q8, w = W.make_q(21, 3)
    cand = W.make_candidates(21, 3, 8, 16, n_dup=2, n_pad=1, n_oob=1)
    return pool, cache, q8, w, cand


def test_sparse_logits_equal_dense_at_mapped_positions():
    pool, cache, q8, w, cand = _tiny_hier()
    for sbk, cbs in ((64, 64), (16, 64), (8, 16)):
        si, end = O.expand_candidates(cand, None, pool.ctx_lens, cbs, sbk)
        sp = O.sparse_logits_decode(q8, w, cache, 64, pool.block_table, None, si, end, sbk)
        dense = O.paged_decode_logits(q8, w, cache, 64, pool.block_table, pool.ctx_lens, 1)
        for r in range(3):
            for c in range(sp.shape[1]):
                if c < end[r]:
                    assert sp[r, c] == dense[r, O.sparse_column_token(si[r], c, sbk)]
                else:
                    assert sp[r, c] == -np.inf


def test_sparse_topk_equals_dense_masked_topk():
    pool, cache, q8, w, cand = _tiny_hier()
    for k in (64, 300, 2048):
        si, end = O.expand_candidates(cand, None, pool.ctx_lens, 64, 64)
        sp = O.sparse_logits_decode(q8, w, cache, 64, pool.block_table, None, si, end, 64)
        for r in range(3):
            cols, pos = O.sparse_topk_remap_row(sp[r], int(end[r]), si[r], 0, 64, k)
            ref = O.dense_masked_topk_row(sp[r], int(end[r]), si[r], 0, int(pool.ctx_lens[r]), 64, k)
            m = min(k, int(end[r]))
            assert np.all(pos[m:] == -1) and np.all(ref[m:] == -1)
            assert set(pos[:m].tolist()) == set(ref[:m].tolist())
            for c, p in zip(cols[:m], pos[:m]):
                assert O.sparse_column_token(si[r], int(c), 64) == p


def test_sparse_remap_golden_with_ks():
    # hand-worked rows whose request starts at ks = 2 SBK and 3 SBK ([V41] 实现拆解 item 3, rows metadata)
    with open(os.path.join(GOLDEN, "sparse_remap.json")) as f:
        spec = json.load(f)
    for c in spec["cases"]:
        si, end = O.expand_candidates_row(c["cand"], c["ks"], c["ke"], c["cand_block_size"], c["sbk"])
        assert list(si) == c["sparse_idx"] and end == c["end"], c["note"]
        vals = np.zeros(len(si) * c["sbk"])
        for col, v in c["scores"].items():
            vals[int(col)] = v
        cols, pos = O.sparse_topk_remap_row(vals, end, si, c["ks"], c["sbk"], c["k"])
        assert list(cols) == c["cols"], c["note"]
        assert list(pos) == c["positions"], c["note"]


def test_sparse_logits_prefill_one_hot_closed_form():
    # one live head / dim / token: the only finite non-zero column is the one that maps onto the token
    sbk, S = 8, 64
    q8 = np.zeros((1, 64, 128), dtype=np.uint8)
    w = np.zeros((1, 64), dtype=np.float32)
    k8 = np.zeros((S, 128), dtype=np.uint8)
    ks = np.ones(S, dtype=np.float32)
    q8[0, 9, 17] = e4m3_encode(3.0)[()]
    w[0, 9] = 0.5
    k8[43, 17] = e4m3_encode(-1.5)[()]
    ks[43] = 0.25
    si = np.array([[5, 2, 6, 6]])         # sparse blocks of 8 tokens: column 3 -> token 43
    out = O.sparse_logits_prefill(q8, w, k8, ks, si, np.array([20]), sbk)
    want = np.full(32, -np.inf)
    want[:20] = 0.0
    want[3] = 0.5 * 3.0 * -1.5 * 0.25
    assert np.array_equal(out[0], want)
    # the same token through another column: block 5 at column 11 when listed second
    out = O.sparse_logits_prefill(q8, w, k8, ks, np.array([[2, 5, 6, 6]]), np.array([32]), sbk)
    assert out[0, 11] == want[3] and np.count_nonzero(out[0]) == 1


def test_sparse_logits_prefill_equal_dense_at_mapped_positions():
    # rows of a prefill chunk whose requests start at ks > 0: every valid sparse column equals the
    # dense prefill logit of its absolute token; columns past end are -inf
    rng = np.random.default_rng(8)
    S, T = 700, 6
    k = rng.standard_normal((S, 128)).astype(np.float32)
    k8, kscale = O.k_quant(k)
    q8, w = W.make_q(8, T)
    for sbk, cbs in ((64, 64), (16, 64), (8, 32)):
        row_ks = np.array([0, sbk, 3 * sbk, 128, 2 * sbk, 5 * sbk])
        row_ke = np.array([700, 650, 400, 300, 2 * sbk + 1, 700])
        cand = rng.integers(-1, 12, (T, 8))
        si, end = O.expand_candidates(cand, row_ks, row_ke, cbs, sbk)
        sp = O.sparse_logits_prefill(q8, w, k8, kscale, si, end, sbk)
        dense = O.mqa_logits(q8, w, k8, kscale, row_ks, row_ke)
        assert np.count_nonzero(end) >= T // 2
        for r in range(T):
            for c in range(sp.shape[1]):
                if c < end[r]:
                    tok = O.sparse_column_token(si[r], c, sbk)
                    assert row_ks[r] <= tok < row_ke[r]
                    assert sp[r, c] == dense[r, tok]
                else:
                    assert sp[r, c] == -np.inf


def test_sparse_topk_equals_dense_masked_topk_with_ks():
    # prefill rows with ks > 0: the remapped selection equals the dense-masked selection over [ks, ke)
    rng = np.random.default_rng(9)
    S, T = 900, 4
    k = rng.standard_normal((S, 128)).astype(np.float32)
    k8, kscale = O.k_quant(k)
    q8, w = W.make_q(9, T)
    row_ks = np.array([64, 192, 320, 128])
    row_ke = np.array([900, 700, 899, 129])
    cand = rng.integers(-1, 14, (T, 8))
    si, end = O.expand_candidates(cand, row_ks, row_ke, 64, 64)
    sp = O.sparse_logits_prefill(q8, w, k8, kscale, si, end, 64)
    for kk in (16, 100, 600):
        for r in range(T):
            cols, pos = O.sparse_topk_remap_row(sp[r], int(end[r]), si[r], int(row_ks[r]), 64, kk)
            ref = O.dense_masked_topk_row(sp[r], int(end[r]), si[r], int(row_ks[r]), int(row_ke[r]), 64, kk)
            m = min(kk, int(end[r]))
            assert np.all(pos[m:] == -1) and np.all(ref[m:] == -1)
            assert set(pos[:m].tolist()) == set(ref[:m].tolist())
            for c, p in zip(cols[:m], pos[:m]):
                assert O.sparse_column_token(si[r], int(c), 64) - row_ks[r] == p
