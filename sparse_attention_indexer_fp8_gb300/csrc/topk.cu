// a5 idx_topk and a9 idx_sparse_topk_remap: per-row radix selection of the k
// largest scores with -1 fill.
//
// "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", opening section: the scorer keeps
// the 2048 highest-scoring history tokens; data-flow item 2: the result is an
// int32 table with -1 for empty entries. The V4.1 review ("实现拆解" item 3)
// runs the same selection over the bf16 sparse logits and then maps each chosen
// sparse column back to its request-local position; here that remap is the
// selection's store step.
//
// Design: one block per row (1024 threads, one block per SM; or 512 threads and
// two blocks per SM when there are many rows of at most 64K columns, so one
// block's barrier-bound phases overlap the other's passes). Scores are mapped to
// order-preserving 32-bit keys and selected by three radix digits (10, 11 and 11
// bits). With more rows than blocks in flight, each block asks for the row one
// wave ahead to be staged in L2. Level 0 histograms the row from global memory
// (or takes the histogram the scoring kernel accumulated); a second pass over
// the row keeps only the elements at or above the threshold digit (bucket A, in
// shared memory) and counts the second digit of those tied with it. The second
// threshold comes from that histogram, the third from one pass over A, and one
// block scan of per-thread (above, tied) counts places every key above the
// threshold key and exactly the number still missing of those equal to it, so
// normally the row is read from global memory once or twice. When bucket A
// overflows its shared-memory buffer, the later levels re-read global memory
// with a prefix filter instead (correct for any input, slower) and reserve
// output slots with warp-aggregated shared-memory counters. The output is a set
// in no particular order.
#include <type_traits>

#include "common.cuh"

namespace idx {

// bit 1: a fused slot conversion produced a slot beyond int32 (written as -1)
__device__ unsigned int g_topk_error = 0;

namespace {

constexpr int kBins = 2048;      // bins of the second and third digits (11 bits each)
constexpr int kBins0 = 1024;     // bins of the first digit (the top 10 key bits)
// Block configurations: 1024 threads and one block per SM for rows of any
// length; 512 threads and two blocks per SM for many shorter rows (prefill
// chunks), so one block's barrier-bound phases overlap the other's passes.
template <int kT>
struct TopkCfg {
  static constexpr int kCapA = kT == 1024 ? 12288 : 6144;  // level-0 hits, above or tied
  static constexpr int kCapB = 4096;                        // level-1 ties (from bucket A)
  static constexpr int kStageBytes = kT * 16 * 4;           // level-0 staging: 16 keys per thread
  // bucket B is first written at level 1, after the staging area's last use
  static constexpr int kUnionBytes = kCapB * 8 > kStageBytes ? kCapB * 8 : kStageBytes;
  static constexpr int kSmemDyn = kCapA * 8 + kUnionBytes;
};
constexpr int kMaxK = 4096;

struct TopkParams {
  const void* logits;
  int64_t ld;
  const int32_t* row_ks;   // plain: range start (NULL = 0); remap: ks of the position base
  const int32_t* row_ke;   // plain: range end
  const int32_t* end;      // remap: range is [0, end[r])
  const int32_t* si;       // remap: sparse block ids
  int64_t ld_si;
  int sbk;
  int k;
  int32_t* out;
  int64_t ld_out;
  int32_t* cols;           // remap: optional chosen columns
  int64_t ld_cols;
  uint32_t* hist;          // optional: precomputed first-digit histogram per row (kBins0 each)
  float* vals;             // optional: the selected scores (fp32), -inf for empty slots
  int64_t ld_vals;
  const int32_t* cand_idx; // merge: shard-local index of every candidate, -1 = empty
  int64_t ld_ci;
  const int32_t* shard_off;  // merge: first global position of each shard (NULL = 0)
  int64_t ld_off;          // merge: row stride of shard_off (0 = one vector for every row)
  int pos_stride;          // merge: global distance between a shard's consecutive positions
  int k_local;             // merge: candidates per shard
  int n_cand;              // merge: candidates per row (shards * k_local)
  // optional slot conversion of the request-local outputs (plain and remap modes):
  // slot = block_table[req(r), v / block_size] * block_span + v % block_size
  int32_t* slots;          // NULL = none
  int64_t ld_slots;
  const int32_t* row_to_req;  // NULL: row r belongs to request r
  const int32_t* bt;
  int64_t ld_bt;
  int block_size;
  int block_span;
  int rows;
  int ahead;               // rows in flight at once (one per SM): the row a wave later is
                           // moved into L2 while this one is selected (0 = off)
};

// What a row selects from and what its outputs mean.
enum Mode : int {
  kPlain = 0,   // columns [ks, ke) of a score row -> request-local indices s - ks
  kRemap = 1,   // sparse columns [0, end) -> request-local positions through the sparse blocks
  kMerge = 2    // candidate lists of several shards -> global positions, empty entries last
};

// The columns [lo, hi) that row `row` selects from.
template <int kMode>
__device__ __forceinline__ void row_range(const TopkParams& p, int row, int64_t& lo, int64_t& hi) {
  if constexpr (kMode == kRemap) {
    lo = 0;
    hi = __ldg(p.end + row);
  } else if constexpr (kMode == kMerge) {
    lo = 0;
    hi = p.n_cand;
  } else {
    lo = p.row_ks ? __ldg(p.row_ks + row) : 0;
    hi = __ldg(p.row_ke + row);
  }
}

template <bool kBf16>
__device__ __forceinline__ uint32_t key_at(const void* row, int64_t c) {
  if constexpr (kBf16) {
    return f32_key(static_cast<uint32_t>(__ldg(static_cast<const uint16_t*>(row) + c)) << 16);
  } else {
    return f32_key(__float_as_uint(__ldg(static_cast<const float*>(row) + c)));
  }
}

// Digits of the key, most significant first: bits 31-22, 21-11, 10-0.
__device__ __forceinline__ int digit(uint32_t key, int level) {
  return level == 0 ? static_cast<int>(key >> 22)
                    : (level == 1 ? static_cast<int>((key >> 11) & 0x7FF)
                                  : static_cast<int>(key & 0x7FF));
}

// True when the bits of `key` above `level` equal those of `prefix`.
__device__ __forceinline__ bool prefix_match(uint32_t key, uint32_t prefix, int level) {
  if (level == 0) return true;
  const uint32_t mask = level == 1 ? 0xFFC00000u : 0xFFFFF800u;
  return (key & mask) == (prefix & mask);
}

// Warp-aggregated slot reservation: returns this lane's slot (valid if pred).
__device__ __forceinline__ int warp_reserve(int* counter, bool pred) {
  const unsigned m = __ballot_sync(0xFFFFFFFFu, pred);
  if (m == 0) return 0;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(0xFFFFFFFFu, base, leader);
  return base + __popc(m & ((1u << lane) - 1u));
}

struct Shared {
  uint32_t hist[2][kBins];
  int warp_tot[32];
  int n_out;      // entries written so far
  int n_a;        // entries offered to bucket A
  int n_b;        // entries offered to bucket B
  int n_tie;      // tickets drawn at the last level
  int thr;
  int need;
  int32_t sel[kMaxK];  // columns chosen so far, in slot order; the outputs are written from them
};

// Finds the digit `thr` at which the running count of larger digits reaches
// `need`; sets sh.thr and reduces sh.need to what must come from bucket `thr`.
template <int kThreads, int nbins, typename S>
__device__ void find_threshold(S& sh, const uint32_t* hist) {
  const int need = sh.need;                // read before any thread can update it
  constexpr int per = nbins / kThreads;    // 1, 2 or 4 (nbins is 1024 or 2048)
  static_assert(per >= 1 && per * kThreads == nbins, "bins per thread");
  const int tid = threadIdx.x;
  int c[per];
  int local = 0;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    c[j] = static_cast<int>(hist[nbins - 1 - (tid * per + j)]);
    local += c[j];
  }
  // exclusive scan of `local` over threads (descending bin order)
  const int lane = tid & 31;
  const int warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) sh.warp_tot[warp] = incl;
  __syncthreads();
  // every warp scans the 32 warp totals itself (no second barrier)
  const int wt = lane < kThreads / 32 ? sh.warp_tot[lane] : 0;
  int wi = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
    if (lane >= o) wi += n;
  }
  const int warp_before = __shfl_sync(0xFFFFFFFFu, wi - wt, warp);
  int before = warp_before + incl - local;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    if (before < need && before + c[j] >= need) {
      sh.thr = nbins - 1 - (tid * per + j);
      sh.need = need - before;
    }
    before += c[j];
  }
  __syncthreads();
}

__device__ __forceinline__ void store_one(Shared& sh, int slot, int64_t col) {
  sh.sel[slot] = static_cast<int32_t>(col);
}

// One selection pass at `level` over a source of (key, column) pairs.
// Elements matching the prefix with digit > thr are stored; digit == thr are
// handed to the next level (appended to `next_keys/next_cols` if room, and
// counted into `next_hist`), or, at the last level, stored while tickets last.
__device__ __forceinline__ void visit(const TopkParams& p, Shared& sh, int row, int64_t lo,
                                      int64_t base_blk, int level, uint32_t prefix, bool valid,
                                      uint32_t key, int64_t col, uint32_t* next_keys,
                                      int32_t* next_cols, int* next_n, int next_cap,
                                      uint32_t* next_hist) {
  const bool in = valid && prefix_match(key, prefix, level);
  const int d = in ? digit(key, level) : -1;
  const int thr = sh.thr;
  // most elements fall below the threshold digit: skip the reservations warp-wide
  if (!__any_sync(0xFFFFFFFFu, d >= thr)) return;
  const bool above = in && d > thr;
  const bool tie = in && d == thr;
  const int s = warp_reserve(&sh.n_out, above);
  if (above && s < p.k) store_one(sh, s, col);
  if (level < 2) {
    if (next_keys) {
      const int t = warp_reserve(next_n, tie);
      if (tie && t < next_cap) {
        next_keys[t] = key;
        next_cols[t] = static_cast<int32_t>(col);
      }
    }
    if (tie) atomicAdd(&next_hist[digit(key, level + 1)], 1u);
  } else {
    const int t = warp_reserve(&sh.n_tie, tie);
    if (tie && t < sh.need) {
      const int slot = atomicAdd(&sh.n_out, 1);
      if (slot < p.k) store_one(sh, slot, col);
    }
  }
}

// Calls f(valid, column, key) for every column of [lo, hi), uniformly across
// every warp of the block (f may use warp collectives). The aligned middle is
// read with 16-byte loads, four per thread in flight; the unaligned head and
// tail (fewer than one vector each) are read element by element.
template <int kThreads, bool kBf16, typename F>
__device__ __forceinline__ void sweep_row(const void* rowp, int64_t lo, int64_t hi, F&& f) {
  constexpr int kVec = kBf16 ? 8 : 4;
  constexpr int kEsz = kBf16 ? 2 : 4;
  constexpr int kUnroll = 4;
  const int tid = threadIdx.x;
  const uintptr_t base = reinterpret_cast<uintptr_t>(rowp);
  int64_t a1 = lo + (kVec - static_cast<int64_t>(((base / kEsz) + lo) % kVec)) % kVec;
  if (a1 > hi) a1 = hi;
  const int64_t nvec = (hi - a1) / kVec;
  const int64_t a2 = a1 + nvec * kVec;
  // head [lo, a1) and tail [a2, hi): at most 2 * (kVec - 1) elements
  {
    const int nh = static_cast<int>(a1 - lo);
    const int nt = static_cast<int>(hi - a2);
    const bool valid = tid < nh + nt;
    const int64_t c = tid < nh ? lo + tid : a2 + (tid - nh);
    f(valid, c, valid ? key_at<kBf16>(rowp, c) : 0u);
  }
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(rowp) + a1 * kEsz);
  // columns and vector indices fit in int32 (rows hold fewer than 2^31 columns)
  constexpr int kStep = kThreads * kUnroll;
  const int nv = static_cast<int>(nvec);
  const int col0 = static_cast<int>(a1);
  auto step = [&](int v0, auto check) {
    constexpr bool kCheck = decltype(check)::value;
    uint4 r[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int v = v0 + j * kThreads + tid;
      r[j] = (!kCheck || v < nv) ? __ldg(vp + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int v = v0 + j * kThreads + tid;
      const bool valid = !kCheck || v < nv;
      const int c = col0 + v * kVec;
      const uint32_t w[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
      for (int e = 0; e < kVec; ++e) {
        uint32_t key;
        if constexpr (kBf16) {
          key = f32_key(((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
        } else {
          key = f32_key(w[e]);
        }
        f(valid, c + e, key);
      }
    }
  };
  const int nfull = nv / kStep * kStep;
  for (int v0 = 0; v0 < nfull; v0 += kStep) step(v0, std::false_type{});
  if (nfull < nv) step(nfull, std::true_type{});
}

// Exclusive prefix sum of v over the warp; *total receives the warp's sum.
__device__ __forceinline__ int warp_excl_scan(int v, int* total) {
  const int lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  *total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  return incl - v;
}

// The level-0 pass over the aligned body of the row. A key is a hit when it is
// at least the smallest key of the threshold digit (so above it or tied with
// it); only hits are kept, appended to bucket A with their columns, and the
// second digit of every tie (a hit of the threshold digit thr0) is counted into
// sh.hist[1] as it is found. Each thread tests the
// 16 elements it loaded into a bit mask and parks the loaded words in its own
// slots of the warp's staging area; one warp scan reserves bucket slots for all
// hits, and each thread then walks only its own set bits (a few per warp at the
// usual hit rate of a few per cent), turning just those into keys.
// The test: when the threshold is a non-negative value (the usual case: the
// 2048 best of thousands of scores) the order-preserving key of a bit pattern u
// is at least tie_lo exactly when u, read as a signed integer, is at least
// tie_lo without its sign bit (negative values and negative NaNs fall below,
// positive NaNs above +inf, as in the key order), so an element costs one
// integer compare; otherwise the key itself is compared.
template <int kThreads, bool kBf16>
__device__ __forceinline__ void level0_collect(Shared& sh, const void* rowp, int64_t a1, int64_t nvec,
                                               uint32_t tie_lo, uint32_t thr0, uint32_t* keys_a,
                                               int32_t* cols_a, uint4* stage) {
  constexpr int kVec = kBf16 ? 8 : 4;
  constexpr int kEsz = kBf16 ? 2 : 4;
  constexpr int kUnroll = kBf16 ? 2 : 4;
  constexpr int kPer = kVec * kUnroll;  // 16 elements per thread per step
  constexpr int kStep = kThreads * kUnroll;  // vectors per step
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  uint4* mine = stage + (tid >> 5) * (kPer / 4) * 32 + lane;  // slot m of this lane: mine[32 * m]
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(rowp) + a1 * kEsz);
  // columns and vector indices fit in int32 (rows hold fewer than 2^31 columns)
  const int nv = static_cast<int>(nvec);
  const int col0 = static_cast<int>(a1);
  const int32_t t_raw = static_cast<int32_t>(tie_lo & 0x7FFFFFFFu);
  // element e of a loaded vector as fp32 bits (bf16: the 16-bit pattern in the upper half)
  auto bits_of = [](const uint32_t (&w)[4], int e) -> uint32_t {
    if constexpr (kBf16) {
      return (e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16);
    } else {
      return w[e];
    }
  };
  // one step: kUnroll vectors per thread; kCheck only for the last, partial step
  auto step = [&](int v0, auto check, auto fast) {
    constexpr bool kCheck = decltype(check)::value;
    constexpr bool kFast = decltype(fast)::value;
    uint4 r[kUnroll];
    uint32_t hit = 0;
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int v = v0 + j * kThreads + tid;
      const bool ok = !kCheck || v < nv;
      r[j] = ok ? __ldg(vp + v) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
      for (int e = 0; e < kVec; ++e) {
        const uint32_t u = bits_of(w, e);
        const bool is_hit = kFast ? static_cast<int32_t>(u) >= t_raw : f32_key(u) >= tie_lo;
        if (ok && is_hit) hit |= 1u << (j * kVec + e);
      }
    }
    int tot;
    int slot = warp_excl_scan(__popc(hit), &tot);
    if (tot == 0) return;
#pragma unroll
    for (int m = 0; m < kUnroll; ++m) mine[32 * m] = r[m];
    int base = 0;
    if (lane == 0) base = atomicAdd(&sh.n_a, tot);
    slot += __shfl_sync(0xFFFFFFFFu, base, 0);
    // the staged words are this thread's own: program order is the only ordering needed
    const uint32_t* mk = reinterpret_cast<const uint32_t*>(mine);
    const int cbase = col0 + (v0 + tid) * kVec;  // column of this thread's first element
    while (hit) {
      const int i = __ffs(hit) - 1;
      hit &= hit - 1;
      uint32_t u;
      if constexpr (kBf16) {
        const uint32_t wd = mk[(i >> 3) * 128 + ((i & 7) >> 1)];
        u = (i & 1) ? (wd & 0xFFFF0000u) : (wd << 16);
      } else {
        u = mk[(i >> 2) * 128 + (i & 3)];
      }
      const uint32_t key = f32_key(u);
      if (slot < TopkCfg<kThreads>::kCapA) {
        keys_a[slot] = key;
        cols_a[slot] = cbase + (i / kVec) * (kThreads * kVec) + i % kVec;
      }
      if ((key >> 22) == thr0) atomicAdd(&sh.hist[1][(key >> 11) & 0x7FFu], 1u);
      ++slot;
    }
  };
  const int nfull = nv / kStep * kStep;
  if (tie_lo >= 0x80000000u) {
    for (int v0 = 0; v0 < nfull; v0 += kStep) step(v0, std::false_type{}, std::true_type{});
    if (nfull < nv) step(nfull, std::true_type{}, std::true_type{});
  } else {
    for (int v0 = 0; v0 < nfull; v0 += kStep) step(v0, std::false_type{}, std::false_type{});
    if (nfull < nv) step(nfull, std::true_type{}, std::false_type{});
  }
}

// Score of column c as fp32.
template <bool kBf16>
__device__ __forceinline__ float value_at(const void* row, int64_t c) {
  if constexpr (kBf16) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const uint16_t*>(row) + c)) << 16);
  } else {
    return __ldg(static_cast<const float*>(row) + c);
  }
}

// The physical slot of request-local position v of row `row` (the conversion of
// idx_req_to_global_slots), -1 for v < 0 or a block index past the table row.
__device__ __forceinline__ int32_t slot_of(const TopkParams& p, int row, int32_t v) {
  if (v < 0) return -1;
  const int64_t lb = v / p.block_size;
  if (lb >= p.ld_bt) return -1;
  const int64_t req = p.row_to_req ? __ldg(p.row_to_req + row) : row;
  const int64_t s = static_cast<int64_t>(__ldg(p.bt + req * p.ld_bt + lb)) * p.block_span + v % p.block_size;
  if (s < 0 || s > INT32_MAX) {
    atomicOr(&g_topk_error, 2u);
    return -1;
  }
  return static_cast<int32_t>(s);
}

// Writes the row's outputs from the chosen columns sh.sel[0, m): mode-specific
// indices (and optionally columns and scores), -1 / -inf in the unused slots.
// In merge mode, candidates without a position are dropped and the remaining
// entries are compacted to the front in slot order.
// Writes output slots s0 + e * kThreads + tid (e < kB, slot < K) of row `row`
// from the chosen columns sel[0, m); the slots past m are empty. A slot takes
// the mode's index (request-local, or the remapped position), optionally the
// physical slot, the column and the score; -1 / -inf for an empty slot. Every
// lookup of the batch (sparse-block id, score, block-table entry) is issued
// before any of its stores. Sparse-block ids below n_si_s come from si_s.
template <int kThreads, int kB, bool kBf16, int kMode>
__device__ __forceinline__ void emit_batch(const TopkParams& p, const int32_t* sel, const int32_t* si_s,
                                           int n_si_s, int row, int64_t lo, int64_t base_blk,
                                           const void* rowp, int s0, int m) {
  const int K = p.k;
  const int tid = threadIdx.x;
  int32_t c[kB], o[kB], sl[kB];
  float v[kB];
#pragma unroll
  for (int e = 0; e < kB; ++e) {
    const int s = s0 + e * kThreads + tid;
    c[e] = s < m ? sel[s] : -1;
  }
#pragma unroll
  for (int e = 0; e < kB; ++e) {
    o[e] = -1;
    v[e] = -__int_as_float(0x7f800000);
    if (c[e] >= 0) {
      if constexpr (kMode == kRemap) {
        const int b = c[e] / p.sbk;
        const int32_t blk = b < n_si_s ? si_s[b] : __ldg(p.si + row * p.ld_si + b);
        o[e] = static_cast<int32_t>((blk - base_blk) * p.sbk + c[e] % p.sbk);
      } else {
        o[e] = static_cast<int32_t>(c[e] - lo);
      }
      if (p.vals) v[e] = value_at<kBf16>(rowp, c[e]);
    }
  }
  if (p.slots) {
#pragma unroll
    for (int e = 0; e < kB; ++e) sl[e] = slot_of(p, row, o[e]);
  }
#pragma unroll
  for (int e = 0; e < kB; ++e) {
    const int s = s0 + e * kThreads + tid;
    if (s < K) {
      p.out[row * p.ld_out + s] = o[e];
      if (p.slots) p.slots[row * p.ld_slots + s] = sl[e];
      if (kMode == kRemap && p.cols) p.cols[row * p.ld_cols + s] = c[e];
      if (p.vals) p.vals[row * p.ld_vals + s] = v[e];
    }
  }
}

template <int kThreads, bool kBf16, int kMode>
__device__ __forceinline__ void write_outputs(const TopkParams& p, Shared& sh, int row, int64_t lo,
                                              const void* rowp, int m) {
  const int tid = threadIdx.x;
  const int K = p.k;
  const float ninf = -__int_as_float(0x7f800000);
  int32_t* out = p.out + row * p.ld_out;
  float* vals = p.vals ? p.vals + row * p.ld_vals : nullptr;
  if constexpr (kMode != kMerge) {
    const int64_t base_blk = (kMode == kRemap && p.row_ks) ? __ldg(p.row_ks + row) / p.sbk : 0;
    constexpr int kB = 4;
    for (int s0 = 0; s0 < K; s0 += kB * kThreads) {
      emit_batch<kThreads, kB, kBf16, kMode>(p, sh.sel, nullptr, 0, row, lo, base_blk, rowp, s0, m);
    }
  } else {
    // each thread owns kMaxK / kThreads consecutive slots; one block scan orders the valid ones
    constexpr int kPer = kMaxK / kThreads;
    int32_t g[kPer];
    float v[kPer];
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = tid * kPer + e;
      g[e] = -1;
      v[e] = ninf;
      if (i < m) {
        const int c = sh.sel[i];
        const int32_t idx = __ldg(p.cand_idx + row * p.ld_ci + c);
        if (idx >= 0) {
          const int32_t off = p.shard_off ? __ldg(p.shard_off + row * p.ld_off + c / p.k_local) : 0;
          g[e] = off + idx * p.pos_stride;
          v[e] = value_at<false>(rowp, c);
          ++cnt;
        }
      }
    }
    const int lane = tid & 31, warp = tid >> 5;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += n;
    }
    __syncthreads();  // sh.warp_tot may still be read by the last threshold search
    if (lane == 31) sh.warp_tot[warp] = incl;
    __syncthreads();
    int before = incl - cnt;
    for (int w = 0; w < warp; ++w) before += sh.warp_tot[w];
    int total = 0;
    for (int w = 0; w < kThreads / 32; ++w) total += sh.warp_tot[w];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      if (g[e] >= 0) {
        if (before < K) {
          out[before] = g[e];
          if (vals) vals[before] = v[e];
        }
        ++before;
      }
    }
    for (int i = total + tid; i < K; i += kThreads) {
      out[i] = -1;
      if (vals) vals[i] = ninf;
    }
  }
}

template <bool kBf16, int kMode, int kThreads>
__global__ void __launch_bounds__(kThreads, 1024 / kThreads) topk_kernel(const TopkParams p) {
  constexpr int kCapA = TopkCfg<kThreads>::kCapA;
  constexpr int kCapB = TopkCfg<kThreads>::kCapB;
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  uint32_t* keys_a = reinterpret_cast<uint32_t*>(dyn);
  int32_t* cols_a = reinterpret_cast<int32_t*>(dyn + kCapA * 4);
  // bucket B and the level-0 staging area share one region (used one after the other)
  uint32_t* keys_b = reinterpret_cast<uint32_t*>(dyn + kCapA * 8);
  int32_t* cols_b = reinterpret_cast<int32_t*>(dyn + kCapA * 8 + kCapB * 4);
  uint4* stage = reinterpret_cast<uint4*>(dyn + kCapA * 8);

  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t base_blk = 0;
  // the workspace histogram is requested before the row's bounds, so the two
  // lookups overlap (plain loads: this kernel clears the words after reading them)
  constexpr int kH0 = kBins0 / kThreads;
  uint32_t* gh = p.hist ? p.hist + static_cast<int64_t>(row) * kBins0 : nullptr;
  uint32_t h0[kH0];
#pragma unroll
  for (int j = 0; j < kH0; ++j) h0[j] = gh ? gh[j * kThreads + tid] : 0u;
  int64_t lo, hi;
  row_range<kMode>(p, row, lo, hi);
  const int64_t n = hi > lo ? hi - lo : 0;
  // More rows than SMs: the row that will most likely run on this SM next (one
  // wave later) is moved into L2 now, by the lanes of warp 0 in 16 KB pieces,
  // so its passes read L2 instead of waiting on DRAM.
  if (p.ahead > 0 && tid < 32 && row + p.ahead < p.rows) {
    constexpr int kEsz = kBf16 ? 2 : 4;
    const int nr = row + p.ahead;
    int64_t nlo, nhi;
    row_range<kMode>(p, nr, nlo, nhi);
    if (nhi > nlo) {
      const uint8_t* nb = static_cast<const uint8_t*>(p.logits) + (static_cast<int64_t>(nr) * p.ld + nlo) * kEsz;
      const uint8_t* b0 = reinterpret_cast<const uint8_t*>((reinterpret_cast<uintptr_t>(nb) + 15) & ~uintptr_t(15));
      const uint8_t* b1 = reinterpret_cast<const uint8_t*>(
          (reinterpret_cast<uintptr_t>(nb) + (nhi - nlo) * kEsz) & ~uintptr_t(15));
      for (const uint8_t* q = b0 + tid * 16384; q < b1; q += 32 * 16384) {
        const int64_t left = b1 - q;
        bulk_prefetch_l2(q, static_cast<uint32_t>(left < 16384 ? left : 16384));
      }
    }
  }
  const int K = p.k;
  const void* rowp = kBf16
      ? static_cast<const void*>(static_cast<const uint16_t*>(p.logits) + row * p.ld)
      : static_cast<const void*>(static_cast<const float*>(p.logits) + row * p.ld);

  if (n <= K) {
    // every visible column is kept, in column order
    if (gh) {
      for (int i = tid; i < kBins0; i += kThreads) gh[i] = 0;
    }
    for (int i = tid; i < n; i += kThreads) sh.sel[i] = static_cast<int32_t>(lo + i);
    __syncthreads();
    write_outputs<kThreads, kBf16, kMode>(p, sh, row, lo, rowp, static_cast<int>(n));
    return;
  }

  for (int i = tid; i < kBins; i += kThreads) {
    sh.hist[0][i] = 0;
    sh.hist[1][i] = 0;
  }
  if (tid == 0) {
    sh.n_out = 0;
    sh.n_a = 0;
    sh.n_b = 0;
    sh.n_tie = 0;
    sh.need = K;
  }
  if (gh) {
    // first digit counted by the kernel that wrote the scores (the same bins
    // this thread just cleared); the workspace is handed back zeroed
#pragma unroll
    for (int j = 0; j < kH0; ++j) {
      sh.hist[0][j * kThreads + tid] = h0[j];
      gh[j * kThreads + tid] = 0;
    }
  }
  __syncthreads();
  if (!gh) {
    // level-0 histogram straight from global memory
    sweep_row<kThreads, kBf16>(rowp, lo, hi, [&](bool valid, int64_t, uint32_t key) {
      if (valid) atomicAdd(&sh.hist[0][key >> 22], 1u);
    });
    __syncthreads();
  }
  find_threshold<kThreads, kBins0>(sh, sh.hist[0]);
  const uint32_t thr0 = static_cast<uint32_t>(sh.thr);

  // level 0: every key at or above the threshold digit goes to bucket A, and
  // the second digit of every key tied on the first is counted on the way
  {
    constexpr int kVec = kBf16 ? 8 : 4;
    constexpr int kEsz = kBf16 ? 2 : 4;
    const uint32_t tie_lo = thr0 << 22;
    const uintptr_t base = reinterpret_cast<uintptr_t>(rowp);
    int64_t a1 = lo + (kVec - static_cast<int64_t>(((base / kEsz) + lo) % kVec)) % kVec;
    if (a1 > hi) a1 = hi;
    const int64_t nvec = (hi - a1) / kVec;
    const int64_t a2 = a1 + nvec * kVec;
    // unaligned head [lo, a1) and tail [a2, hi), element by element
    {
      const int nh = static_cast<int>(a1 - lo);
      const int nt = static_cast<int>(hi - a2);
      const bool valid = tid < nh + nt;
      const int64_t c = tid < nh ? lo + tid : a2 + (tid - nh);
      const uint32_t key = valid ? key_at<kBf16>(rowp, c) : 0u;
      const bool h = valid && key >= tie_lo;
      const int s = warp_reserve(&sh.n_a, h);
      if (h && s < kCapA) {
        keys_a[s] = key;
        cols_a[s] = static_cast<int32_t>(c);
      }
      if (h && (key >> 22) == thr0) atomicAdd(&sh.hist[1][(key >> 11) & 0x7FFu], 1u);
    }
    level0_collect<kThreads, kBf16>(sh, rowp, a1, nvec, tie_lo, thr0, keys_a, cols_a, stage);
    __syncthreads();
  }
  const int na0 = sh.n_a;
  if (na0 <= kCapA) {
    // Bucket A holds every hit. The two remaining digits are found over the
    // tied keys (the second from the histogram of the pass, the third from one
    // pass over A), then one block scan of per-thread (above, tied) counts
    // gives each chosen key its output slot: every key above the threshold key
    // and `need` of those equal to it.
    for (int i = tid; i < kBins; i += kThreads) sh.hist[0][i] = 0;  // level 0's search is done
    find_threshold<kThreads, kBins>(sh, sh.hist[1]);
    const uint32_t p1 = (thr0 << 11) | static_cast<uint32_t>(sh.thr);
    for (int i = tid; i < na0; i += kThreads) {
      const uint32_t key = keys_a[i];
      if ((key >> 11) == p1) atomicAdd(&sh.hist[0][key & 0x7FFu], 1u);
    }
    __syncthreads();
    find_threshold<kThreads, kBins>(sh, sh.hist[0]);
    const uint32_t tkey = (p1 << 11) | static_cast<uint32_t>(sh.thr);
    // a workspace histogram that does not match the scores can leave any count
    // here; the clamp keeps every slot inside the row's outputs
    const int need = min(max(sh.need, 0), K);
    // this thread's keys of A are i = tid, tid + kThreads, ...; the scan runs in thread order
    uint32_t cnt = 0;  // above | tied << 16 (each total is at most kCapA)
    for (int i = tid; i < na0; i += kThreads) {
      const uint32_t key = keys_a[i];
      cnt += key > tkey ? 1u : (key == tkey ? 0x10000u : 0u);
    }
    const int lane = tid & 31;
    const int warp = tid >> 5;
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.warp_tot[warp] = static_cast<int>(incl);
    __syncthreads();
    // every warp scans the warp totals itself
    const uint32_t wt = lane < kThreads / 32 ? static_cast<uint32_t>(sh.warp_tot[lane]) : 0u;
    uint32_t wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += y;
    }
    const uint32_t before = __shfl_sync(0xFFFFFFFFu, wi - wt, warp) + (incl - cnt);
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, wi, 31);
    int a = static_cast<int>(before & 0xFFFFu);
    int t = static_cast<int>(before >> 16);
    for (int i = tid; i < na0; i += kThreads) {
      const uint32_t key = keys_a[i];
      if (key > tkey) {
        const int s = a + min(t, need);
        ++a;
        if (s < K) sh.sel[s] = cols_a[i];
      } else if (key == tkey) {
        if (t < need && a + t < K) sh.sel[a + t] = cols_a[i];
        ++t;
      }
    }
    __syncthreads();
    const int a_tot = static_cast<int>(total & 0xFFFFu);
    const int t_tot = static_cast<int>(total >> 16);
    write_outputs<kThreads, kBf16, kMode>(p, sh, row, lo, rowp, min(K, a_tot + min(need, t_tot)));
    return;
  }
  // More hits than bucket A holds: classify the row again from global memory,
  // storing the chosen directly and keeping as many ties as fit (the second
  // digit's histogram is counted again by this pass).
  __syncthreads();
  for (int i = tid; i < kBins; i += kThreads) sh.hist[1][i] = 0;
  if (tid == 0) sh.n_a = 0;
  __syncthreads();
  sweep_row<kThreads, kBf16>(rowp, lo, hi, [&](bool valid, int64_t c, uint32_t key) {
    visit(p, sh, row, lo, base_blk, 0, 0u, valid, key, c, keys_a, cols_a, &sh.n_a, kCapA, sh.hist[1]);
  });
  uint32_t prefix = thr0 << 22;
  __syncthreads();
  for (int i = tid; i < kBins; i += kThreads) sh.hist[0][i] = 0;  // free since level 0 is done
  find_threshold<kThreads, kBins>(sh, sh.hist[1]);
  prefix |= static_cast<uint32_t>(sh.thr) << 11;

  // level 1: from bucket A when it held every tie, else global memory with a prefix filter
  const bool a_ok = sh.n_a <= kCapA;
  const int na = sh.n_a;
  if (a_ok) {
    for (int base = 0; base < na; base += kThreads) {
      const int i = base + tid;
      const bool valid = i < na;
      visit(p, sh, row, lo, base_blk, 1, prefix, valid, valid ? keys_a[i] : 0u,
                    valid ? cols_a[i] : 0, keys_b, cols_b, &sh.n_b, kCapB, sh.hist[0]);
    }
  } else {
    sweep_row<kThreads, kBf16>(rowp, lo, hi, [&](bool valid, int64_t c, uint32_t key) {
      visit(p, sh, row, lo, base_blk, 1, prefix, valid, key, c, keys_b, cols_b, &sh.n_b,
                    kCapB, sh.hist[0]);
    });
  }
  __syncthreads();
  find_threshold<kThreads, kBins>(sh, sh.hist[0]);
  prefix |= static_cast<uint32_t>(sh.thr);

  // level 2: every remaining candidate shares the full key prefix; take the bucket
  // above the threshold and exactly `need` of the tied keys
  const int nb = sh.n_b;
  if (nb <= kCapB) {
    for (int base = 0; base < nb; base += kThreads) {
      const int i = base + tid;
      const bool valid = i < nb;
      visit(p, sh, row, lo, base_blk, 2, prefix, valid, valid ? keys_b[i] : 0u,
                    valid ? cols_b[i] : 0, nullptr, nullptr, nullptr, 0, nullptr);
    }
  } else if (a_ok) {
    for (int base = 0; base < na; base += kThreads) {
      const int i = base + tid;
      const bool valid = i < na;
      visit(p, sh, row, lo, base_blk, 2, prefix, valid, valid ? keys_a[i] : 0u,
                    valid ? cols_a[i] : 0, nullptr, nullptr, nullptr, 0, nullptr);
    }
  } else {
    sweep_row<kThreads, kBf16>(rowp, lo, hi, [&](bool valid, int64_t c, uint32_t key) {
      visit(p, sh, row, lo, base_blk, 2, prefix, valid, key, c, nullptr, nullptr, nullptr,
                    0, nullptr);
    });
  }
  // With exact counts exactly k columns were chosen. A histogram that does not
  // match the scores (a misused workspace) can leave a short row: it is
  // completed with -1 by the output pass.
  __syncthreads();
  write_outputs<kThreads, kBf16, kMode>(p, sh, row, lo, rowp, min(sh.n_out, K));
}

// Rows of at most kShortMax columns (the sparse rows of the V4.1 path: 64
// candidate blocks of 64 tokens). One 256-thread block per row, several rows in
// flight on every SM. Each thread keeps its 16 keys in registers (16-byte loads
// where the row is aligned), so nothing but the histograms and the chosen
// columns goes through shared memory. The key has 16 significant bits for bf16
// scores and 32 for fp32; its 8-bit digits are resolved most significant first
// (two levels for bf16, four for fp32), each level histogramming only the keys
// that share the digits above. The last level fixes the threshold key and how
// many of the keys equal to it are kept. One block-wide scan of per-thread
// counts (above, tied) in column order then gives every chosen key its output
// slot directly: the chosen columns come out in column order, and among keys
// equal to the threshold the lowest columns are kept. The row's sparse-block
// ids are staged in shared memory with the row loads, so the output pass has
// no dependent global loads (except for the fused slot conversion).
constexpr int kShortThreads = 256;
constexpr int kShortMax = 4096;
constexpr int kShortPer = kShortMax / kShortThreads;  // row elements per thread
constexpr int kShortSi = 1024;                        // sparse-block ids staged per row
constexpr int kEmitBatch = 8;                         // output slots per thread per batch

struct ShortShared {
  int32_t sel[kMaxK];  // chosen columns, in slot order
  int32_t si[kShortSi];
  uint32_t hist[2][256];
  uint32_t tot[4][kShortThreads / 32];  // per chunk and warp: packed (above, tied) counts
  int warp_tot[32];
  int thr;
  int need;
};

// Order-preserving key of a raw score: the upper 16 bits of the fp32 key for
// bf16 (its lower 16 bits are a function of the sign), the fp32 key otherwise.
template <bool kBf16>
__device__ __forceinline__ uint32_t short_key(uint32_t raw) {
  return kBf16 ? f32_key(raw << 16) >> 16 : f32_key(raw);
}

template <bool kBf16, int kMode>
__global__ void __launch_bounds__(kShortThreads, 4) topk_short_kernel(const TopkParams p) {
  __shared__ ShortShared sh;
  constexpr int kVec = kBf16 ? 8 : 4;         // elements per 16-byte load
  constexpr int kEsz = kBf16 ? 2 : 4;
  constexpr int kChunks = kShortPer / kVec;   // 2 or 4
  constexpr int kSpan = kVec * kShortThreads; // elements per chunk
  constexpr int kLevels = kBf16 ? 2 : 4;      // 8-bit digits of the key
  constexpr int kWarps = kShortThreads / 32;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  int64_t lo, hi;
  row_range<kMode>(p, row, lo, hi);
  const int n = hi > lo ? static_cast<int>(hi - lo) : 0;
  const int K = p.k;
  const void* rowp = kBf16
      ? static_cast<const void*>(static_cast<const uint16_t*>(p.logits) + row * p.ld)
      : static_cast<const void*>(static_cast<const float*>(p.logits) + row * p.ld);
  const int64_t base_blk = (kMode == kRemap && p.row_ks) ? __ldg(p.row_ks + row) / p.sbk : 0;
  // Elements [0, lim) of the window may be read. A sparse row's window starts at
  // column 0, so its loads need not wait for end[row]: every column below
  // min(ld, kShortMax) lies inside the row.
  const int lim = kMode == kRemap ? static_cast<int>(p.ld < kShortMax ? p.ld : kShortMax) : n;
  int n_si_s = 0;
  if constexpr (kMode == kRemap) {
    const int nb = (lim + p.sbk - 1) / p.sbk;
    const int ns = static_cast<int>(nb < p.ld_si ? nb : p.ld_si);
    if (ns <= kShortSi) {
      n_si_s = ns;
      for (int i = tid; i < ns; i += kShortThreads) sh.si[i] = __ldg(p.si + row * p.ld_si + i);
    }
  }
  if (p.hist) {
    // the workspace histogram is not used for rows this short; it is handed back zeroed
    uint32_t* g = p.hist + static_cast<int64_t>(row) * kBins0;
    for (int i = tid; i < kBins0; i += kShortThreads) g[i] = 0;
  }
  if (n <= K) {
    // every visible column is kept, in column order
    for (int i = tid; i < n; i += kShortThreads) sh.sel[i] = static_cast<int32_t>(lo + i);
    __syncthreads();
    for (int s0 = 0; s0 < K; s0 += kEmitBatch * kShortThreads) {
      emit_batch<kShortThreads, kEmitBatch, kBf16, kMode>(p, sh.sel, sh.si, n_si_s, row, lo, base_blk, rowp, s0, n);
    }
    return;
  }
  // key of element h * kSpan + tid * kVec + j at [h * kVec + j]
  uint32_t key[kShortPer];
  {
    const char* wp = static_cast<const char*>(rowp) + lo * kEsz;
    const bool vec = (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0 && p.ld % kVec == 0 && lo % kVec == 0;
    if (vec) {
      // a vector that starts inside [0, lim) ends inside the row
      uint4 r[kChunks];
#pragma unroll
      for (int h = 0; h < kChunks; ++h) {
        const int i0 = h * kSpan + tid * kVec;
        r[h] = i0 < lim ? __ldg(reinterpret_cast<const uint4*>(wp + static_cast<int64_t>(i0) * kEsz))
                        : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int h = 0; h < kChunks; ++h) {
        const uint32_t w[4] = {r[h].x, r[h].y, r[h].z, r[h].w};
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
          const uint32_t raw = kBf16 ? ((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu) : w[j];
          key[h * kVec + j] = short_key<kBf16>(raw);
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < kChunks; ++h) {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
          const int i = h * kSpan + tid * kVec + j;
          uint32_t raw = 0;
          if (i < lim) {
            raw = kBf16 ? static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(wp) + i))
                        : __float_as_uint(__ldg(reinterpret_cast<const float*>(wp) + i));
          }
          key[h * kVec + j] = short_key<kBf16>(raw);
        }
      }
    }
  }
  sh.hist[0][tid] = 0;
  sh.hist[1][tid] = 0;
  if (tid == 0) sh.need = K;
  __syncthreads();
  // digits, most significant first; the threshold key collects them
  uint32_t tkey = 0;
#pragma unroll
  for (int L = 0; L < kLevels; ++L) {
    const int sft = 8 * (kLevels - 1 - L);
    uint32_t* hist = sh.hist[L & 1];
#pragma unroll
    for (int e = 0; e < kShortPer; ++e) {
      const int i = (e / kVec) * kSpan + tid * kVec + (e % kVec);
      // the digits above this level equal those chosen so far (none at level 0)
      const bool in = i < n && (L == 0 || (key[e] >> (sft + 8)) == (tkey >> (sft + 8)));
      if (in) atomicAdd(&hist[(key[e] >> sft) & 0xFFu], 1u);
    }
    __syncthreads();
    find_threshold<kShortThreads, 256>(sh, hist);
    tkey |= static_cast<uint32_t>(sh.thr) << sft;
    // reused two levels down: every read of it ended before find_threshold's last barrier
    hist[tid] = 0;
  }
  const int need = sh.need;  // keys equal to tkey still to take
  // per-thread counts of keys above and equal to the threshold, per chunk,
  // packed as above | tied << 16 (each total is at most kShortMax)
  uint32_t excl[kChunks];
#pragma unroll
  for (int h = 0; h < kChunks; ++h) {
    uint32_t a = 0, t = 0;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int i = h * kSpan + tid * kVec + j;
      if (i < n) {
        a += key[h * kVec + j] > tkey;
        t += key[h * kVec + j] == tkey;
      }
    }
    const uint32_t cnt = a | (t << 16);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.tot[h][warp] = incl;
    excl[h] = incl - cnt;
  }
  __syncthreads();
  {
    // exclusive prefix in column order: earlier chunks, then earlier warps of this chunk
    uint32_t run = 0;
#pragma unroll
    for (int h = 0; h < kChunks; ++h) {
      uint32_t before = 0, total = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t v = sh.tot[h][w];
        before += w < warp ? v : 0u;
        total += v;
      }
      excl[h] += run + before;
      run += total;
    }
  }
#pragma unroll
  for (int h = 0; h < kChunks; ++h) {
    int a = static_cast<int>(excl[h] & 0xFFFFu);
    int t = static_cast<int>(excl[h] >> 16);
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int i = h * kSpan + tid * kVec + j;
      const uint32_t kk = key[h * kVec + j];
      if (i < n) {
        if (kk > tkey) {
          const int s = a + min(t, need);
          ++a;
          if (s < K) sh.sel[s] = static_cast<int32_t>(lo + i);
        } else if (kk == tkey) {
          if (t < need && a + t < K) sh.sel[a + t] = static_cast<int32_t>(lo + i);
          ++t;
        }
      }
    }
  }
  __syncthreads();
  // the keys above the threshold and `need` of those equal to it: exactly K
  for (int s0 = 0; s0 < K; s0 += kEmitBatch * kShortThreads) {
    emit_batch<kShortThreads, kEmitBatch, kBf16, kMode>(p, sh.sel, sh.si, n_si_s, row, lo, base_blk, rowp, s0, K);
  }
}

}  // namespace

unsigned int topk_read_and_clear_error(cudaStream_t stream, cudaError_t* err) {
  unsigned int v = 0;
  const unsigned int zero = 0;
  *err = cudaStreamSynchronize(stream);
  if (*err != cudaSuccess) return 0;
  *err = cudaMemcpyFromSymbol(&v, g_topk_error, sizeof(v));
  if (*err != cudaSuccess) return 0;
  if (v) *err = cudaMemcpyToSymbol(g_topk_error, &zero, sizeof(zero));
  return v;
}

}  // namespace idx

using namespace idx;

namespace {

// The optional workspace holds, per row, the first-digit histogram that the
// logits entry points accumulate when given the same workspace.
idx_status_t attach_hist(const char* fn, TopkParams* p, int rows, void* ws, size_t ws_bytes) {
  if (!ws) return IDX_OK;
  const size_t need = static_cast<size_t>(rows) * kBins0 * sizeof(uint32_t);
  if (ws_bytes < need) {
    return fail(IDX_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes, need);
  }
  if (!aligned(ws, 16)) return fail(IDX_ERR_UNSUPPORTED, "%s: workspace must be 16-byte aligned", fn);
  p->hist = static_cast<uint32_t*>(ws);
  return IDX_OK;
}

// The optional fused slot conversion (the checks of idx_req_to_global_slots).
idx_status_t attach_slots(const char* fn, TopkParams* p, int32_t k, const int32_t* row_to_req,
                          const int32_t* block_table, int64_t ld_bt, int32_t block_size,
                          int32_t block_span, int32_t* slots, int64_t ld_slots) {
  if (!slots) return fail(IDX_ERR_INVALID_ARG, "%s: NULL slots", fn);
  if (!block_table) return fail(IDX_ERR_INVALID_ARG, "%s: NULL block_table", fn);
  if (block_size < 1 || ld_bt < 1) return fail(IDX_ERR_INVALID_ARG, "%s: block_size and ld_bt must be positive", fn);
  if (block_span < block_size) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: block_span %d < block_size %d", fn, block_span, block_size);
  }
  if (ld_slots < k) return fail(IDX_ERR_INVALID_ARG, "%s: ld_slots < k", fn);
  p->slots = slots;
  p->ld_slots = ld_slots;
  p->row_to_req = row_to_req;
  p->bt = block_table;
  p->ld_bt = ld_bt;
  p->block_size = block_size;
  p->block_span = block_span;
  return IDX_OK;
}

template <bool kBf16, int kMode, int kThreads>
idx_status_t launch_topk_cfg(TopkParams p, int rows, int sms, cudaStream_t stream, const char* fn) {
  auto kern = topk_kernel<kBf16, kMode, kThreads>;
  constexpr int smem = TopkCfg<kThreads>::kSmemDyn;
  // 1024 / kThreads blocks per SM: 228 KB of shared memory per SM, 1 KB reserved per block
  static_assert((smem + sizeof(Shared) + 1024) * (1024 / kThreads) <= 233472, "blocks per SM");
  static_assert(smem + sizeof(Shared) <= 232448, "shared memory per block");
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(IDX_ERR_CUDA, "%s: cudaFuncSetAttribute: %s", fn, cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int resident = sms * (1024 / kThreads);  // blocks in flight at once
  p.rows = rows;
  p.ahead = sms > 0 && rows > resident ? resident : 0;
  kern<<<rows, kThreads, smem, stream>>>(p);
  return check_launch(fn);
}

}  // namespace

namespace idx {

bool topk_rows_short(int64_t rows, int64_t max_cols) {
  const int sms = device_sm_count();
  return rows > 0 && max_cols <= kShortMax && sms > 0;
}

}  // namespace idx

namespace {

// Rows of at most kShortMax columns take the short-row kernel; many rows of at
// most 64K columns (prefill chunks) the two-blocks-per-SM configuration;
// anything else one 1024-thread block per SM.
template <bool kBf16, int kMode>
idx_status_t launch_topk(const TopkParams& p, int rows, int64_t max_cols, cudaStream_t stream,
                         const char* fn) {
  const int sms = device_sm_count();
  if constexpr (kMode != kMerge) {
    if (topk_rows_short(rows, max_cols)) {
      // short rows: one 256-thread block per row with the keys in registers,
      // several rows in flight per SM; with one row per SM as well (128-row
      // sparse decode) its short chain beats the 1024-thread block's passes
      TopkParams q = p;
      q.rows = rows;
      q.ahead = 0;
      topk_short_kernel<kBf16, kMode><<<rows, kShortThreads, 0, stream>>>(q);
      return check_launch(fn);
    }
  }
  if (sms > 0 && rows > 2 * sms && max_cols <= 65536) {
    return launch_topk_cfg<kBf16, kMode, 512>(p, rows, sms, stream, fn);
  }
  return launch_topk_cfg<kBf16, kMode, 1024>(p, rows, sms, stream, fn);
}

}  // namespace

namespace {

idx_status_t topk_common(const char* fn, const void* logits, int dtype, int64_t ld,
                         const int32_t* row_ks, const int32_t* row_ke, int32_t rows, int32_t k,
                         int32_t* out, int64_t ld_out, float* vals, int64_t ld_vals, void* ws,
                         size_t ws_bytes, TopkParams& p, cudaStream_t stream) {
  if (rows < 0 || k < 1) return fail(IDX_ERR_INVALID_ARG, "%s: rows < 0 or k < 1", fn);
  if (k > kMaxK) return fail(IDX_ERR_UNSUPPORTED, "%s: k %d exceeds %d", fn, k, kMaxK);
  if (ld_out < k || (vals && ld_vals < k)) return fail(IDX_ERR_INVALID_ARG, "%s: output stride < k", fn);
  if (dtype != IDX_F32 && dtype != IDX_BF16) return fail(IDX_ERR_UNSUPPORTED, "%s: dtype %d", fn, dtype);
  if (rows == 0) return IDX_OK;
  if (!logits || !row_ke || !out) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  idx_status_t st = attach_hist(fn, &p, rows, ws, ws_bytes);
  if (st != IDX_OK) return st;
  p.logits = logits;
  p.ld = ld;
  p.row_ks = row_ks;
  p.row_ke = row_ke;
  p.k = k;
  p.out = out;
  p.ld_out = ld_out;
  p.vals = vals;
  p.ld_vals = ld_vals;
  return dtype == IDX_BF16 ? launch_topk<true, kPlain>(p, rows, ld, stream, fn)
                           : launch_topk<false, kPlain>(p, rows, ld, stream, fn);
}

}  // namespace

extern "C" idx_status_t idx_topk(const void* logits, int dtype, int64_t ld, const int32_t* row_ks,
                                 const int32_t* row_ke, int32_t rows, int32_t k, int32_t* out,
                                 int64_t ld_out, float* vals, int64_t ld_vals, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  TopkParams p{};
  return topk_common("idx_topk", logits, dtype, ld, row_ks, row_ke, rows, k, out, ld_out, vals,
                     ld_vals, ws, ws_bytes, p, stream);
}

extern "C" idx_status_t idx_topk_slots(const void* logits, int dtype, int64_t ld,
                                       const int32_t* row_ks, const int32_t* row_ke, int32_t rows,
                                       int32_t k, int32_t* out, int64_t ld_out,
                                       const int32_t* row_to_req, const int32_t* block_table,
                                       int64_t ld_bt, int32_t block_size, int32_t block_span,
                                       int32_t* slots, int64_t ld_slots, void* ws, size_t ws_bytes,
                                       cudaStream_t stream) {
  const char* fn = "idx_topk_slots";
  TopkParams p{};
  if (rows > 0) {
    idx_status_t st = attach_slots(fn, &p, k, row_to_req, block_table, ld_bt, block_size, block_span,
                                   slots, ld_slots);
    if (st != IDX_OK) return st;
  }
  return topk_common(fn, logits, dtype, ld, row_ks, row_ke, rows, k, out, ld_out, nullptr, 0, ws,
                     ws_bytes, p, stream);
}

namespace {

idx_status_t remap_common(const char* fn, const void* sparse_logits, int dtype, int64_t ld,
                          const int32_t* end, const int32_t* sparse_idx, int64_t ld_si,
                          const int32_t* row_ks, int32_t sbk, int32_t rows, int32_t k,
                          int32_t* col_scratch, int64_t ld_col, int32_t* positions, int64_t ld_pos,
                          void* ws, size_t ws_bytes, TopkParams& p, cudaStream_t stream) {
  if (rows < 0 || k < 1 || sbk < 1) return fail(IDX_ERR_INVALID_ARG, "%s: rows < 0, k < 1 or sbk < 1", fn);
  if (k > kMaxK) return fail(IDX_ERR_UNSUPPORTED, "%s: k %d exceeds %d", fn, k, kMaxK);
  if (ld_pos < k || (col_scratch && ld_col < k)) return fail(IDX_ERR_INVALID_ARG, "%s: output stride < k", fn);
  if (dtype != IDX_F32 && dtype != IDX_BF16) return fail(IDX_ERR_UNSUPPORTED, "%s: dtype %d", fn, dtype);
  if (rows == 0) return IDX_OK;
  if (!sparse_logits || !end || !sparse_idx || !positions) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  idx_status_t st = attach_hist(fn, &p, rows, ws, ws_bytes);
  if (st != IDX_OK) return st;
  p.logits = sparse_logits;
  p.ld = ld;
  p.row_ks = row_ks;
  p.end = end;
  p.si = sparse_idx;
  p.ld_si = ld_si;
  p.sbk = sbk;
  p.k = k;
  p.out = positions;
  p.ld_out = ld_pos;
  p.cols = col_scratch;
  p.ld_cols = ld_col;
  return dtype == IDX_BF16 ? launch_topk<true, kRemap>(p, rows, ld, stream, fn)
                           : launch_topk<false, kRemap>(p, rows, ld, stream, fn);
}

}  // namespace

extern "C" idx_status_t idx_sparse_topk_remap(const void* sparse_logits, int dtype, int64_t ld,
                                              const int32_t* end, const int32_t* sparse_idx,
                                              int64_t ld_si, const int32_t* row_ks, int32_t sbk,
                                              int32_t rows, int32_t k, int32_t* col_scratch,
                                              int64_t ld_col, int32_t* positions, int64_t ld_pos,
                                              void* ws, size_t ws_bytes, cudaStream_t stream) {
  TopkParams p{};
  return remap_common("idx_sparse_topk_remap", sparse_logits, dtype, ld, end, sparse_idx, ld_si,
                      row_ks, sbk, rows, k, col_scratch, ld_col, positions, ld_pos, ws, ws_bytes, p,
                      stream);
}

extern "C" idx_status_t idx_sparse_topk_remap_slots(
    const void* sparse_logits, int dtype, int64_t ld, const int32_t* end, const int32_t* sparse_idx,
    int64_t ld_si, const int32_t* row_ks, int32_t sbk, int32_t rows, int32_t k, int32_t* col_scratch,
    int64_t ld_col, int32_t* positions, int64_t ld_pos, const int32_t* row_to_req,
    const int32_t* block_table, int64_t ld_bt, int32_t block_size, int32_t block_span,
    int32_t* slots, int64_t ld_slots, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const char* fn = "idx_sparse_topk_remap_slots";
  TopkParams p{};
  if (rows > 0) {
    idx_status_t st = attach_slots(fn, &p, k, row_to_req, block_table, ld_bt, block_size, block_span,
                                   slots, ld_slots);
    if (st != IDX_OK) return st;
  }
  return remap_common(fn, sparse_logits, dtype, ld, end, sparse_idx, ld_si, row_ks, sbk, rows, k,
                      col_scratch, ld_col, positions, ld_pos, ws, ws_bytes, p, stream);
}

extern "C" idx_status_t idx_dcp_topk_merge(const float* cand_vals, int64_t ld_v,
                                           const int32_t* cand_idx, int64_t ld_i,
                                           const int32_t* shard_offset, int64_t ld_off,
                                           int32_t n_shards, int32_t pos_stride, int32_t k_local,
                                           int32_t rows, int32_t k, int32_t* out, int64_t ld_out,
                                           float* vals, int64_t ld_vals, cudaStream_t stream) {
  const char* fn = "idx_dcp_topk_merge";
  if (rows < 0 || k < 1 || n_shards < 1 || k_local < 1 || pos_stride < 1) {
    return fail(IDX_ERR_INVALID_ARG,
                "%s: rows < 0, k < 1, n_shards < 1, k_local < 1 or pos_stride < 1", fn);
  }
  if (ld_off != 0 && ld_off < n_shards) return fail(IDX_ERR_INVALID_ARG, "%s: 0 < ld_off < n_shards", fn);
  if (k > kMaxK) return fail(IDX_ERR_UNSUPPORTED, "%s: k %d exceeds %d", fn, k, kMaxK);
  const int64_t n_cand = static_cast<int64_t>(n_shards) * k_local;
  if (n_cand > INT32_MAX / 2) return fail(IDX_ERR_UNSUPPORTED, "%s: too many candidates", fn);
  if (ld_v < n_cand || ld_i < n_cand) return fail(IDX_ERR_INVALID_ARG, "%s: candidate stride < n_shards * k_local", fn);
  if (ld_out < k || (vals && ld_vals < k)) return fail(IDX_ERR_INVALID_ARG, "%s: output stride < k", fn);
  if (rows == 0) return IDX_OK;
  if (!cand_vals || !cand_idx || !out) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  TopkParams p{};
  p.logits = cand_vals;
  p.ld = ld_v;
  p.cand_idx = cand_idx;
  p.ld_ci = ld_i;
  p.shard_off = shard_offset;
  p.ld_off = ld_off;
  p.pos_stride = pos_stride;
  p.k_local = k_local;
  p.n_cand = static_cast<int>(n_cand);
  p.k = k;
  p.out = out;
  p.ld_out = ld_out;
  p.vals = vals;
  p.ld_vals = ld_vals;
  return launch_topk<false, kMerge>(p, rows, n_cand, stream, fn);
}
