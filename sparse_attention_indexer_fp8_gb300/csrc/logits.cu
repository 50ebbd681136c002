// a3 / a4 / a8: FP8 MQA logits on the 5th-generation tensor core.
//
//   logits[t, s] = kscale[s] * sum_{h < 64} w[t, h] * sum_{d < 128} q8[t, h, d] * k8[s, d]
//
// ("DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", "Indexer 内部六步" step 6: the 64
// head dot products collapsed into one score by the per-head weights; step 4:
// all q-side coefficients live in the weights. k is the dequantised cache
// entry, its fp32 scale applied per column.)
//
// One kernel serves the four ways the path reads k:
//   decode dense   - the paged cache through the block table, no gather (the
//                    page's prefill/decode kernel table);
//   decode sparse  - only the candidate sparse blocks of each row (the V4.1
//                    review, "功能与动机" and "实现拆解" item 3);
//   prefill dense  - gathered contiguous k with ragged causal row limits;
//   prefill sparse - gathered k restricted to each row's sparse blocks.
//
// Orientation. A tile is 128 consecutive output columns (tokens). The MMA is
// D[128 x N] += A[128 x 32] * B[N x 32]^T, four times over K = 128, with
// A = the tile's 128 k rows (e4m3, K-major, 128-byte swizzle) and B = the
// group's q (N = 64 heads x NQ query rows, K-major), so the fp32 accumulator
// in tensor memory holds one TOKEN per lane and one (query, head) per column.
// Each epilogue thread therefore owns one token and reduces its 64 head
// columns against the weights in registers: the weighted head sum needs no
// cross-thread traffic and the [rows x 64 heads x tokens] intermediate never
// leaves the SM.
//
// Roles (persistent CTAs; with one or two queries per group, decode and the
// sparse modes, two 192-thread CTAs per SM with one epilogue warpgroup each: two
// independent pipelines per SM stream the cache at a markedly higher rate than
// one; with four queries per group, prefill, one 320-thread CTA per SM with two
// epilogue warpgroups):
//   warp 0     TMA producer: k boxes (one per cache block / sparse block) and
//              their scales into a ring of shared-memory stages, q per group;
//              block-table lookups for the next tile are issued before the
//              wait for a free stage so their latency hides behind it.
//   warp 1     allocates tensor memory; one lane issues tcgen05.mma and
//              commits stage / accumulator barriers (MXFP4 k: the warp first
//              stages the tile's block scales and copies them into tensor
//              memory with tcgen05.cp).
//   warps 2-   epilogue, warpgroups taking tiles in turn: tcgen05.ld of
//              the accumulator, weighted head sum, scale, causal / range mask,
//              coalesced store (fp32 or bf16).
// The flattened (group, tile) sequence is split evenly over the CTAs; every
// role walks the same sequence. Every wait is bounded; on expiry the CTA
// records a device error code and leaves in order.
#include <cuda_bf16.h>

#include <type_traits>

#include "common.cuh"

namespace idx {

namespace {

constexpr int kTile = 128;

constexpr int kKvStageBytes = kTile * kDim;       // 16 KB
constexpr int kScaleStageBytes = 2048;            // up to 16 boxes, each in a 128-byte slot
constexpr uint64_t kTimeoutNs = 2000000000ull;

enum Mode : int { kDecodeDense = 0, kDecodeSparse = 1, kPrefillDense = 2, kPrefillSparse = 3 };

// Bit (1 << w) of g_logits_error: wait site w (1..7) expired. The first
// expiry also records where it happened in g_logits_error_info:
// {site, block, tile ordinal, group, tile, barrier index, parity, 0}.
__device__ unsigned int g_logits_error = 0;
__device__ unsigned int g_logits_error_taken = 0;
__device__ long long g_logits_error_info[8];

struct LogitsParams {
  int mode;
  int n_groups;
  int tiles_per_group;  // modes with a fixed column count; unused for decode dense
  int n_rows;           // q / w / output rows
  int next_n;
  int nq;               // rows per group in the dense modes
  const void* w;
  int w_bf16;
  int64_t ld_w;
  int paged;
  const uint8_t* kv_base;     // cache (paged) or k8 (contiguous)
  int64_t kv_block_stride;    // bytes between cache blocks (paged)
  int unit;             // tokens per k box (cache block, sparse block or 128)
  int scale_slot;       // bytes between the scale boxes of one stage (>= 128)
  int unit_shift;       // log2(unit) (a power of two)
  int slot_shift;       // log2(scale_slot)
  int block_size;
  const int32_t* block_table;
  int64_t ld_bt;
  const int32_t* ctx_lens;
  int S;
  const int32_t* row_ks;
  const int32_t* row_ke;
  const int32_t* sparse_idx;
  int64_t ld_si;
  int n_si;
  const int32_t* end;
  int sbk;
  void* out;
  int out_bf16;
  int64_t ld_out;
  // 1: the scores are stored with an L2 evict-last policy, so the selection that
  // reads them next finds them in L2 rather than behind the evict-first k stream
  int out_keep_l2;
  // optional: per-row histogram of the top 10 key bits of every visible logit
  // (kHistBins uint32 per row), accumulated for the selection's first digit
  uint32_t* hist;
};

constexpr int kHistBins = 1024;  // first selection digit: the top 10 bits of the order-preserving key

// kFp4: k read from the MXFP4 cache (one query per group only). The MMA warp
// copies each tile's block scales into tensor memory ahead of its MMAs; they
// take columns from the accumulators: three accumulator stages, a commit per
// tile, then one 4-column scale slot per k stage and one for q.
template <int NQ, bool kFp4 = false, bool kHist = true>
struct Cfg {
  static_assert(!kFp4 || NQ == 1, "the MXFP4 path serves one query per group");
  static constexpr int N = 64 * NQ;
  // CTAs per SM and epilogue warpgroups per CTA (taking tiles in turn)
  static constexpr int kCtasPerSm = NQ == 4 ? 1 : 2;
  static constexpr int kEpiWG = NQ == 4 ? 2 : 1;
  static constexpr int kEpiWarps = 4 * kEpiWG;
  static constexpr int kThreads = 64 + kEpiWarps * 32;
  // k stages; one query per group without the workspace histogram: the
  // histogram area's shared memory holds a fifth stage instead
  static constexpr int kStages = NQ == 4 ? 8 : (NQ == 1 && !kHist ? 5 : 4);
  static constexpr int kAccStages = NQ == 1 ? (kFp4 ? 3 : 4) : 2;
  // tiles per tcgen05.commit: one commit covers the MMAs of kCommit consecutive
  // tiles (commits are costly next to a 4-MMA tile); one accumulator-ready
  // barrier per commit group
  static constexpr int kCommit = NQ == 1 && !kFp4 ? 2 : 1;
  static constexpr int kAccFull = kAccStages / kCommit;
  // MXFP4: the scale words of k stage s at columns kSfaCol + 4 s .. + 3 (row r of
  // the tile in lane r, column + r / 32), q's (all 1.0) at kSfbCol .. + 3
  static constexpr int kSfaCol = kAccStages * N;
  static constexpr int kSfbCol = kSfaCol + 4 * kStages;
  static constexpr int kTmemCols = kFp4 ? 256 : kAccStages * N;  // 256 or 512 per CTA, 512 per SM
  static_assert(!kFp4 || kSfbCol + 4 <= kTmemCols, "scale columns fit the allocation");
  static constexpr int kQStageBytes = NQ * 64 * kDim;
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kStages * kKvStageBytes;
  static constexpr int kOffScale = kOffQ + 2 * kQStageBytes;
  static constexpr int kOffW = kOffScale + kStages * kScaleStageBytes;
  // per epilogue warp, one query per group: 1024 bins of 16-bit counts
  static constexpr int kHistWords = NQ == 1 && kHist ? kHistBins / 2 : 0;
  static constexpr int kOffHist = kOffW + kEpiWarps * NQ * 64 * 4;
  static constexpr int kOffSf = kOffHist + kEpiWarps * kHistWords * 4;
  // MXFP4: per k stage the tile's 128 scale words as 32 lines of 16 bytes (line m
  // holds rows m, m + 32, m + 64, m + 96), the layout the 32x128b.warpx4
  // tensor-memory copy spreads over the four lane quarters; then one such block
  // of 1.0 scales for q
  static constexpr int kSfLineBytes = kFp4 ? 512 * (kStages + 1) : 0;
  static constexpr int kOffBar = kOffSf + kSfLineBytes;
  static constexpr int kNumBars = 2 * kStages + kAccFull + kAccStages + 4;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448 / kCtasPerSm - 2048, "shared memory budget per CTA");
  static_assert(kTmemCols * kCtasPerSm <= 512, "tensor memory columns per SM");
};

struct Group {
  int row0;    // first q row of the group
  int nq;      // rows in the group
  int req;     // request whose block table is used (paged modes)
  int ncols;   // columns written per row: [0, ncols)
  int tiles;   // 128-column tiles
  int act_lo;  // union of the rows' visible columns: [act_lo, act_hi)
  int act_hi;
};

__device__ __forceinline__ Group load_group(const LogitsParams& p, int g) {
  Group G;
  switch (p.mode) {
    case kDecodeDense: {
      const int L = max(__ldg(p.ctx_lens + g), 0);
      G.row0 = g * p.next_n;
      G.nq = p.next_n;
      G.req = g;
      G.ncols = L;
      G.tiles = (L + kTile - 1) / kTile;
      G.act_lo = 0;
      G.act_hi = L;
      break;
    }
    case kPrefillDense: {
      G.row0 = g * p.nq;
      G.nq = min(p.nq, p.n_rows - G.row0);
      G.req = 0;
      G.ncols = p.S;
      G.tiles = p.tiles_per_group;
      int lo = INT32_MAX, hi = 0;
      for (int j = 0; j < G.nq; ++j) {
        const int ks = p.row_ks ? max(__ldg(p.row_ks + G.row0 + j), 0) : 0;
        const int ke = min(__ldg(p.row_ke + G.row0 + j), p.S);
        if (ke > ks) {
          lo = min(lo, ks);
          hi = max(hi, ke);
        }
      }
      G.act_lo = hi > 0 ? lo : 0;
      G.act_hi = hi;
      break;
    }
    default: {  // sparse modes: one row per group
      G.row0 = g;
      G.nq = 1;
      G.req = p.mode == kDecodeSparse ? g / p.next_n : 0;
      G.ncols = p.n_si * p.sbk;
      G.tiles = p.tiles_per_group;
      G.act_lo = 0;
      G.act_hi = min(max(__ldg(p.end + g), 0), G.ncols);
      break;
    }
  }
  return G;
}

__device__ __forceinline__ bool tile_active(const Group& G, int t) {
  return t * kTile < G.act_hi && t * kTile + kTile > G.act_lo;
}

// Walks this CTA's share of the flattened (group, tile) sequence.
struct Walker {
  int g, t;
  long long left;
  Group G;
  __device__ __forceinline__ void init(const LogitsParams& p, int g0, int t0, long long n) {
    g = g0;
    t = t0;
    left = n;
    if (left > 0) G = load_group(p, g);
  }
  __device__ __forceinline__ void advance(const LogitsParams& p) {
    if (--left <= 0) return;
    if (++t >= G.tiles) {
      do {
        ++g;
        G = load_group(p, g);
      } while (G.tiles == 0);
      t = 0;
    }
  }
};

// Bounded wait. All threads that call it for the same barrier get the same
// answer only if they also agree on abort; callers make the result warp-uniform.
// `ord`, `g`, `t` and `bar_idx` only describe the wait for the error record.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int site, long long ord = -1, int g = -1,
                                         int t = -1, int bar_idx = -1) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      atomicOr(&g_logits_error, 1u << site);
      if (atomicCAS(&g_logits_error_taken, 0u, 1u) == 0u) {
        g_logits_error_info[0] = site;
        g_logits_error_info[1] = blockIdx.x;
        g_logits_error_info[2] = ord;
        g_logits_error_info[3] = g;
        g_logits_error_info[4] = t;
        g_logits_error_info[5] = bar_idx;
        g_logits_error_info[6] = parity;
        g_logits_error_info[7] = 0;
      }
      return false;
    }
  }
}

// Coordinates of one k box: cache block (0 when contiguous) and row inside it.
struct Box {
  int blk;
  int row;
  bool valid;
};

// Box u of tile t of a group whose first row is row0, whose request is req and
// whose rows see the columns [act_lo, act_hi).
__device__ __forceinline__ Box box_at(const LogitsParams& p, int row0, int req, int act_lo,
                                      int act_hi, int t, int u) {
  Box b;
  const int c0 = t * kTile + u * p.unit;
  b.valid = c0 < act_hi && c0 + p.unit > act_lo;
  b.blk = 0;
  b.row = 0;
  if (!b.valid) return b;
  int tok = c0;
  if (p.mode == kDecodeSparse || p.mode == kPrefillSparse) {
    tok = __ldg(p.sparse_idx + static_cast<int64_t>(row0) * p.ld_si + c0 / p.sbk) * p.sbk;
  }
  if (p.paged) {
    b.blk = __ldg(p.block_table + static_cast<int64_t>(req) * p.ld_bt + tok / p.block_size);
    b.row = tok % p.block_size;
  } else {
    b.row = tok;
  }
  return b;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

__device__ __forceinline__ float hsum2(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}

// sum_h w[h] * acc[h] over the 64 head columns of one query (a0: heads 0-31,
// a1: heads 32-63), with the packed two-lane fp32 FMA of sm_100+: half the FMA
// instructions of the scalar form, four independent two-lane accumulators.
// w4(i) returns the weights of heads 4i..4i+3 (registers, or one broadcast
// 16-byte shared-memory load).
template <typename W4Fn>
__device__ __forceinline__ float weighted_head_sum(const uint32_t (&a0)[32], const uint32_t (&a1)[32],
                                                   W4Fn w4) {
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int h = 0; h < 32; h += 4) {
    const float4 w = w4(h >> 2);
    fma2(acc[(h >> 1) & 3], pack2(__uint_as_float(a0[h]), __uint_as_float(a0[h + 1])), pack2(w.x, w.y));
    fma2(acc[((h >> 1) + 1) & 3], pack2(__uint_as_float(a0[h + 2]), __uint_as_float(a0[h + 3])),
         pack2(w.z, w.w));
  }
#pragma unroll
  for (int h = 0; h < 32; h += 4) {
    const float4 w = w4(8 + (h >> 2));
    fma2(acc[(h >> 1) & 3], pack2(__uint_as_float(a1[h]), __uint_as_float(a1[h + 1])), pack2(w.x, w.y));
    fma2(acc[((h >> 1) + 1) & 3], pack2(__uint_as_float(a1[h + 2]), __uint_as_float(a1[h + 3])),
         pack2(w.z, w.w));
  }
  return (hsum2(acc[0]) + hsum2(acc[1])) + (hsum2(acc[2]) + hsum2(acc[3]));
}

template <int NQ, bool kOutBf16, bool kFp4, bool kHist>
__global__ void __launch_bounds__(Cfg<NQ, kFp4, kHist>::kThreads, Cfg<NQ, kFp4, kHist>::kCtasPerSm)
mqa_logits_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                  const __grid_constant__ CUtensorMap map_scale, const LogitsParams p) {
  using C = Cfg<NQ, kFp4, kHist>;
  constexpr int kThreads = C::kThreads;
  constexpr int kEpiWG = C::kEpiWG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* kv_s = smem + C::kOffKv;
  uint8_t* q_s = smem + C::kOffQ;
  uint8_t* sc_s = smem + C::kOffScale;
  float* w_s = reinterpret_cast<float*>(smem + C::kOffW);
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + C::kOffHist);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* acc_full = bars + 2 * C::kStages;
  uint64_t* acc_empty = acc_full + C::kAccFull;
  uint64_t* q_full = acc_empty + C::kAccStages;
  uint64_t* q_empty = q_full + 2;
  uint8_t* sf_lines = smem + C::kOffSf;  // MXFP4 (see Cfg::kSfLineBytes)

  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_g0, s_t0;
  __shared__ long long s_count;
  __shared__ int4 s_tile[2][32];   // producer batches: (group, tile, row0, req)
  __shared__ int2 s_act[2][32];    //                   (act_lo, act_hi)
  __shared__ int s_ntile[2];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      // released by the 4 warps of the epilogue warpgroup that owns the tile, once
      // its accumulator is ready (so the MMAs no longer read the stage)
      mbar_init(&empty[s], 4);
    }
    for (int a = 0; a < C::kAccFull; ++a) mbar_init(&acc_full[a], 1);
    for (int a = 0; a < C::kAccStages; ++a) mbar_init(&acc_empty[a], 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    fence_mbar_init();
    s_abort = 0;
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_kv);
    tma_prefetch_map(&map_scale);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }

  // ---- this CTA's share of the (group, tile) sequence ----
  // Split evenly over the CTAs: [total * b / grid, total * (b + 1) / grid). In
  // dense decode the tile count of a group follows its context length: the last
  // warp walks the lengths 32 groups at a time (the total, then the group that
  // holds this CTA's first tile) while warps 0 and 1 set up the barriers and
  // tensor memory.
  if (p.mode == kDecodeDense) {
    if (warp == kThreads / 32 - 1) {
      auto tiles_of = [&](int g) -> int {
        return g < p.n_groups ? (max(__ldg(p.ctx_lens + g), 0) + kTile - 1) / kTile : 0;
      };
      long long total = 0;
      for (int base = 0; base < p.n_groups; base += 32) {
        int v = tiles_of(base + lane);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        total += v;
      }
      const long long u0 = total * blockIdx.x / gridDim.x;
      const long long u1 = total * (blockIdx.x + 1) / gridDim.x;
      if (lane == 0) {
        s_count = u1 - u0;
        s_g0 = 0;
        s_t0 = 0;
      }
      __syncwarp();
      long long run = 0;
      for (int base = 0; base < p.n_groups && u1 > u0; base += 32) {
        const int v = tiles_of(base + lane);
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += n;
        }
        const long long hi = run + incl;
        const bool hit = v > 0 && hi - v <= u0 && u0 < hi;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, hit);
        if (m) {
          if (lane == __ffs(m) - 1) {
            s_g0 = base + lane;
            s_t0 = static_cast<int>(u0 - (hi - v));
          }
          break;
        }
        run += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
  } else if (threadIdx.x == 0) {
    const long long total = static_cast<long long>(p.n_groups) * p.tiles_per_group;
    const long long u0 = total * blockIdx.x / gridDim.x;
    const long long u1 = total * (blockIdx.x + 1) / gridDim.x;
    s_count = u1 - u0;
    s_g0 = p.tiles_per_group > 0 ? static_cast<int>(u0 / p.tiles_per_group) : 0;
    s_t0 = p.tiles_per_group > 0 ? static_cast<int>(u0 % p.tiles_per_group) : 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const long long count = s_count;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // =========================== TMA producer ===========================
    // Boxes are prepared a batch at a time, one lane per box: lane 0 walks the
    // next batch of active tiles and publishes it in shared memory, then every
    // lane fetches the sparse-index / block-table entries of its own box. The
    // next batch is fetched before the current one is issued, so those dependent
    // loads overlap with the waits for free stages instead of serialising.
    // Decode reads every k box once (evict first) and keeps q; a prefill chunk
    // re-reads the same k rows for every query group (keep them in L2) while
    // each group's q is read by one or two CTAs.
    const bool prefill = p.mode == kPrefillDense || p.mode == kPrefillSparse;
    const uint64_t pol_kv = prefill ? l2_policy_evict_last() : l2_policy_evict_first();
    const uint64_t pol_q = prefill ? l2_policy_evict_first() : l2_policy_evict_last();
    const int upt = kTile / p.unit;  // boxes per tile, 1..16
    const int tpb = 32 / upt;        // tiles per batch
    // bytes a box moves from global memory (the FP4 tensor map counts the packed
    // bytes it reads, not the padded bytes it writes to shared memory)
    const uint32_t box_bytes = static_cast<uint32_t>(p.unit) * (kFp4 ? kMxTokenBytes : kTokenBytes);
    int st = 0;
    uint32_t ph = 0;
    int qs = 0;
    uint32_t qph = 0;
    int q_group = -1;
    bool ok = true;
    Walker W;
    W.init(p, s_g0, s_t0, count);
    auto fill = [&](int buf) {  // lane 0
      int n = 0;
      while (W.left > 0 && n < tpb) {
        if (tile_active(W.G, W.t)) {
          s_tile[buf][n] = make_int4(W.g, W.t, W.G.row0, W.G.req);
          s_act[buf][n] = make_int2(W.G.act_lo, W.G.act_hi);
          ++n;
        }
        W.advance(p);
      }
      s_ntile[buf] = n;
    };
    auto coords = [&](int buf) -> Box {
      Box b;
      b.valid = false;
      b.blk = 0;
      b.row = 0;
      const int ti = lane / upt;
      if (ti < s_ntile[buf]) {
        const int4 tl = s_tile[buf][ti];
        const int2 act = s_act[buf][ti];
        b = box_at(p, tl.z, tl.w, act.x, act.y, tl.y, lane - ti * upt);
      }
      return b;
    };
    auto issue_batch = [&](int buf, const Box& bx) -> bool {
      const int n = s_ntile[buf];
      for (int ti = 0; ti < n; ++ti) {
        const int4 tl = s_tile[buf][ti];
        if (tl.x != q_group) {
          bool got = true;
          if (lane == 0) got = wait_bar(&q_empty[qs], qph ^ 1u, abort_flag, 1u, -1, tl.x, tl.y, qs);
          got = __shfl_sync(0xFFFFFFFFu, got, 0);
          if (!got) return false;
          if (lane == 0) {
            mbar_arrive_expect_tx(&q_full[qs], C::kQStageBytes);
            tma_load_3d(q_s + qs * C::kQStageBytes, &map_q, &q_full[qs], 0, 0, tl.z, pol_q);
          }
          q_group = tl.x;
          if (++qs == 2) {
            qs = 0;
            qph ^= 1u;
          }
        }
        bool got = true;
        if (lane == 0) got = wait_bar(&empty[st], ph ^ 1u, abort_flag, 2u, -1, tl.x, tl.y, st);
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) return false;
        const bool mine = (lane / upt == ti) && bx.valid;
        const unsigned vm = __ballot_sync(0xFFFFFFFFu, mine);
        if (lane == 0) mbar_arrive_expect_tx(&full[st], __popc(vm) * box_bytes);
        __syncwarp();
        if (mine) {
          const int u = lane - ti * upt;
          tma_load_3d(kv_s + st * kKvStageBytes + u * p.unit * kDim, &map_kv, &full[st], 0, bx.row,
                      bx.blk, pol_kv);
          tma_load_2d(sc_s + st * kScaleStageBytes + u * p.scale_slot, &map_scale, &full[st],
                      bx.row, bx.blk, pol_kv);
        }
        if (++st == C::kStages) {
          st = 0;
          ph ^= 1u;
        }
      }
      return true;
    };
    if (lane == 0) fill(0);
    __syncwarp();
    Box cur = coords(0);
    int buf = 0;
    while (ok && s_ntile[buf] > 0) {
      if (lane == 0) fill(buf ^ 1);
      __syncwarp();
      const Box nxt = coords(buf ^ 1);
      ok = issue_batch(buf, cur);
      cur = nxt;
      buf ^= 1;
      __syncwarp();
    }
    // drain: wait for every load still in flight before the CTA can exit
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
        // the most recent phase of stage s was issued with parity ph (s < st) or ph ^ 1
        const uint32_t par = s < st ? ph : (ph ^ 1u);
        uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&full[s], par) && global_timer_ns() - t0 < kTimeoutNs) {
        }
      }
      for (int i = 0; i < 2; ++i) {
        const uint32_t par = i < qs ? qph : (qph ^ 1u);
        uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&q_full[i], par) && global_timer_ns() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp == 1) {
    // =========================== MMA issuer ===========================
    // One lane issues the tensor-core work. For MXFP4 tiles the whole warp
    // first moves the tile's scale words into the copy layout: lane m gathers
    // the words of rows m, m + 32, m + 64, m + 96 into one 16-byte line, and the
    // issuing lane then copies the 32 lines into tensor memory
    // (tcgen05.cp.32x128b.warpx4: line m lands in lane m of every lane quarter,
    // so row r finds its word in lane r, column r / 32, where the block-scaled
    // MMA reads it) ahead of the tile's MMAs. Copy and MMAs are issued by one
    // thread and execute in issue order.
    constexpr uint32_t idesc = idesc_e4m3_f32(kTile, C::N);
    int st = 0, as = 0, qs = 0;
    uint32_t ph = 0, aph = 0, qph = 0;
    int q_group = -1;
    long long ai = 0;  // active tiles issued
    Walker W;
    W.init(p, s_g0, s_t0, count);
    // e4m3 k: only lane 0 runs the loop. MXFP4 k: the whole warp does (it stages
    // the scales); lane 0 waits and the answer is shared with the warp.
    auto wait0 = [&](uint64_t* bar, uint32_t par, unsigned site, int idx) -> bool {
      if constexpr (!kFp4) {
        return wait_bar(bar, par, abort_flag, site, ai, W.g, W.t, idx);
      } else {
        bool got = true;
        if (lane == 0) got = wait_bar(bar, par, abort_flag, site, ai, W.g, W.t, idx);
        return __shfl_sync(0xFFFFFFFFu, got, 0);
      }
    };
    if constexpr (kFp4) {
      // q's scales: 1.0 (E8M0 code 127) everywhere, copied once before the first MMA
      *reinterpret_cast<uint4*>(sf_lines + C::kStages * 512 + lane * 16) =
          make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tmem_cp_32x128b_warpx4(tmem_base + static_cast<uint32_t>(C::kSfbCol),
                               lines_desc(smem_u32(sf_lines + C::kStages * 512)));
      }
    }
    bool ok = kFp4 || lane == 0;
    while (W.left > 0 && ok) {
      if (tile_active(W.G, W.t)) {
        if (W.g != q_group) {
          if (q_group >= 0) {
            if (lane == 0) umma_commit(&q_empty[qs]);
            if (++qs == 2) {
              qs = 0;
              qph ^= 1u;
            }
          }
          if (!wait0(&q_full[qs], qph, 3u, qs)) break;
          q_group = W.g;
        }
        if constexpr (kFp4) {
          // every lane reads the loaded scale words, so every lane waits for the stage
          const bool got = wait_bar(&full[st], ph, abort_flag, 4u, ai, W.g, W.t, st);
          if (!__all_sync(0xFFFFFFFFu, got)) break;
          const uint8_t* sc = sc_s + st * kScaleStageBytes;
          uint32_t v[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            // row r is word r % unit of scale box r / unit (powers of two: shifts, no division)
            const int r = lane + 32 * q4;
            v[q4] = *reinterpret_cast<const uint32_t*>(sc + ((r >> p.unit_shift) << p.slot_shift) +
                                                       ((r & (p.unit - 1)) << 2));
          }
          *reinterpret_cast<uint4*>(sf_lines + st * 512 + lane * 16) = make_uint4(v[0], v[1], v[2], v[3]);
          fence_proxy_async_smem();  // the copy reads these lines through the async proxy
          __syncwarp();
        } else {
          if (!wait0(&full[st], ph, 4u, st)) break;
        }
        if (!wait0(&acc_empty[as], aph ^ 1u, 5u, as)) break;
        if (lane == 0) {
          tc_fence_after();
          const uint64_t a_desc = sw128_kmajor_desc(smem_u32(kv_s + st * kKvStageBytes));
          const uint64_t b_desc = sw128_kmajor_desc(smem_u32(q_s + qs * C::kQStageBytes));
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as * C::N);
          if constexpr (kFp4) {
            // the FP4 tile sits in shared memory as 16-element groups padded to 16
            // bytes, so a K block of 32 elements spans 32 bytes exactly as e4m3 does;
            // K block k takes byte k of every scale word
            constexpr uint32_t mx = idesc_mx_e2m1_e4m3(kTile, C::N);
            const uint32_t sfa = tmem_base + static_cast<uint32_t>(C::kSfaCol + 4 * st);
            const uint32_t sfb = tmem_base + static_cast<uint32_t>(C::kSfbCol);
            tmem_cp_32x128b_warpx4(sfa, lines_desc(smem_u32(sf_lines + st * 512)));
#pragma unroll
            for (int k = 0; k < kDim / 32; ++k) {
              umma_mx_e2m1_e4m3(d_tmem, a_desc + 2 * k, b_desc + 2 * k,
                                idesc_with_scale_ids(mx, static_cast<uint32_t>(k), static_cast<uint32_t>(k)),
                                sfa, sfb, k > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kDim / 32; ++k) {
              // +32 bytes along K inside the 128-byte swizzled rows = +2 in the >>4 address field
              umma_e4m3(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, k > 0 ? 1u : 0u);
            }
          }
          if ((ai + 1) % C::kCommit == 0) umma_commit(&acc_full[(ai / C::kCommit) % C::kAccFull]);
        }
        if constexpr (kFp4) __syncwarp();
        ++ai;
        if (++st == C::kStages) {
          st = 0;
          ph ^= 1u;
        }
        if (++as == C::kAccStages) {
          as = 0;
          aph ^= 1u;
        }
      }
      W.advance(p);
    }
    if (lane == 0) {
      // an unfinished commit group (odd tile count) still needs its commit
      if (ai % C::kCommit != 0) umma_commit(&acc_full[((ai - 1) / C::kCommit) % C::kAccFull]);
      if (q_group >= 0) umma_commit(&q_empty[qs]);
    }
    __syncwarp();
  } else {
    // =========================== epilogue ===========================
    // kEpiWG warpgroups take the commit groups of active tiles in turn, so
    // consecutive tiles overlap their TMEM-load / FMA / store latency chains.
    // Ring positions follow from the active-tile ordinal. Every accumulator
    // stage and every accumulator-ready barrier belongs to one warpgroup for the
    // whole kernel (kAccFull is a multiple of kEpiWG). The commit of group
    // cg + kAccFull needs an accumulator stage that group cg's first tile
    // releases, so a barrier never runs ahead of the one wait per group below.
    static_assert(C::kAccFull % kEpiWG == 0, "accumulator barriers per warpgroup");
    const int ew = warp - 2;
    const int wg = ew / 4;
    const int quarter = warp & 3;  // tensor-memory lanes this warp may read
    const int trow = quarter * 32 + lane;
    // this thread's token row inside a stage's scale boxes: word trow % unit of box trow / unit
    const int sc_off = ((trow >> p.unit_shift) << p.slot_shift) + ((trow & (p.unit - 1)) << 2);
    const uint64_t pol_out = l2_policy_evict_last();
    float* wsm = w_s + ew * NQ * 64;
    // private histogram of this warp's visible logits for the current group;
    // flushed to the row's global histogram when the warp moves to another group
    uint32_t* wh = hist_s + ew * C::kHistWords;
    const bool do_hist = C::kHistWords > 0 && p.hist != nullptr;
    int hist_row = -1;
    int hist_tiles = 0;  // tiles counted since the last flush: 16-bit bins hold < 2048 tiles
    if (do_hist) {
      for (int i = lane; i < C::kHistWords; i += 32) wh[i] = 0;
      __syncwarp();
    }
    auto flush_hist = [&]() {
      if (!do_hist || hist_row < 0) return;
      __syncwarp();
      uint32_t* g = p.hist + static_cast<int64_t>(hist_row) * kHistBins;
      for (int i = lane; i < C::kHistWords; i += 32) {
        const uint32_t v = wh[i];
        if (v) {
          if (v & 0xFFFFu) atomicAdd(g + 2 * i, v & 0xFFFFu);
          if (v >> 16) atomicAdd(g + 2 * i + 1, v >> 16);
          wh[i] = 0;
        }
      }
      __syncwarp();
      hist_row = -1;
      hist_tiles = 0;
    };
    // Per-CTA tile ordinals fit in int: a CTA's share of any cache or score
    // matrix that fits in device memory is far below 2^31 tiles.
    int ai = 0;  // active tiles seen
    // A warp waits a commit group's accumulator-ready barrier once, at the
    // group's first tile. Waiting again at the second tile would be unsafe: once
    // the first tile's accumulator is released the MMA warp may already commit
    // the group two ahead (an unpaired last tile of the range commits at once)
    // to the same barrier, moving it two phases past this wait's parity.
    int waited_cg = -1;
    int cur_g = -1;
    int lim_lo[NQ], lim_hi[NQ];
    using OutT = typename std::conditional<kOutBf16, __nv_bfloat16, float>::type;
    OutT* orow[NQ];  // output row of each query of the current group
    // one query per group: its 64 weights live in registers for the whole group
    constexpr bool kRegW = NQ == 1;
    float wreg[kRegW ? 64 : 1];
    const float ninf = -__int_as_float(0x7f800000);
    // The CTA's (group, tile) range, a group at a time. Active tiles come in
    // the producer's and MMA warp's order (ordinal ai); this warpgroup visits
    // only the tiles of its own commit groups, and fills the inactive tiles of
    // the range (those outside the group's visible columns) whose index is
    // congruent to it, so every tile costs a warp no bookkeeping unless it is
    // that warp's to process.
    int g = s_g0;
    int tb = s_t0;
    long long left = count;
    bool stop = false;
    while (left > 0 && !stop) {
      const Group G = load_group(p, g);
      const int te = static_cast<int>(min(static_cast<long long>(G.tiles), tb + left));
      left -= te - tb;
      // active tiles of the group within [tb, te): the tiles that meet [act_lo, act_hi)
      const int ta0 = max(G.act_lo / kTile, tb);
      const int ta1 = max(min((G.act_hi + kTile - 1) / kTile, te), ta0);
      const int nact = ta1 - ta0;
      // first active tile of this warpgroup's commit groups
      const int cg_first = ai / C::kCommit;
      const int skip = (wg - cg_first % kEpiWG + kEpiWG) % kEpiWG;
      int oi = skip == 0 ? 0 : (cg_first + skip) * C::kCommit - ai;
      if (oi < nact && g != cur_g) {
        flush_hist();
        cur_g = g;
        __syncwarp();
        for (int i = lane; i < NQ * 64; i += 32) {
          const int j = i >> 6;
          float v = 0.f;
          if (j < G.nq) {
            const int64_t off = static_cast<int64_t>(G.row0 + j) * p.ld_w + (i & 63);
            v = p.w_bf16
                    ? __uint_as_float(static_cast<uint32_t>(
                                          __ldg(reinterpret_cast<const uint16_t*>(p.w) + off))
                                      << 16)
                    : __ldg(reinterpret_cast<const float*>(p.w) + off);
          }
          wsm[i] = v;
        }
        __syncwarp();
        if constexpr (kRegW) {
#pragma unroll
          for (int i = 0; i < 64; ++i) wreg[i] = wsm[i];
        }
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          int lo = 0, hi = 0;
          if (j < G.nq) {
            if (p.mode == kDecodeDense) {
              hi = min(max(G.ncols - p.next_n + j + 1, 0), G.ncols);
            } else if (p.mode == kPrefillDense) {
              lo = p.row_ks ? max(__ldg(p.row_ks + G.row0 + j), 0) : 0;
              hi = min(__ldg(p.row_ke + G.row0 + j), p.S);
            } else {
              hi = G.act_hi;
            }
          }
          lim_lo[j] = lo;
          lim_hi[j] = hi;
          orow[j] = reinterpret_cast<OutT*>(p.out) + static_cast<int64_t>(G.row0 + j) * p.ld_out;
        }
      }
      // inactive tiles of the range: -inf
      for (int t = tb; t < te; ++t) {
        if (t >= ta0 && t < ta1) {
          t = ta1 - 1;
          continue;
        }
        const int c = t * kTile + trow;
        if (t % kEpiWG != wg || c >= G.ncols) continue;
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          if (j < G.nq) {
            const int64_t o = static_cast<int64_t>(G.row0 + j) * p.ld_out + c;
            if constexpr (kOutBf16) {
              reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(ninf);
            } else {
              reinterpret_cast<float*>(p.out)[o] = ninf;
            }
          }
        }
      }
      while (oi < nact && !stop) {
        const int a = ai + oi;
        const int t = ta0 + oi;
        const int c = t * kTile + trow;
        const int st = a % C::kStages;
        const uint32_t ph = static_cast<uint32_t>((a / C::kStages) & 1);
        const int as = a % C::kAccStages;
        const int cg = a / C::kCommit;
        const int af = cg % C::kAccFull;
        const uint32_t afph = static_cast<uint32_t>((cg / C::kAccFull) & 1);
        bool got = wait_bar(&full[st], ph, abort_flag, 6u, a, g, t, st);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          stop = true;
          break;
        }
        // the token's fp32 scale (the MXFP4 block scales were applied by the MMA)
        const float scale = kFp4 ? 1.0f : *reinterpret_cast<const float*>(sc_s + st * kScaleStageBytes + sc_off);
        if (cg != waited_cg) {
          got = wait_bar(&acc_full[af], afph, abort_flag, 7u, a, g, t, af);
          if (!__all_sync(0xFFFFFFFFu, got)) {
            stop = true;
            break;
          }
          waited_cg = cg;
        }
        tc_fence_after();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // the MMAs of this tile are done with the stage
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(as * C::N);
        // The weighted head sum of every query is reduced into registers first;
        // the accumulator is handed back to the MMA warp before any global store,
        // so the release (which orders this thread's earlier writes) never waits
        // on the logits stores.
        float logit[NQ];
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          logit[j] = 0.f;
          if (j < G.nq) {
            uint32_t a0[32], a1[32];
            tmem_ld_x32(taddr + j * 64, a0);
            tmem_ld_x32(taddr + j * 64 + 32, a1);
            tmem_wait_ld(a0);
            reg_fence(a1);
            float sum;
            if constexpr (kRegW) {
              sum = weighted_head_sum(a0, a1, [&](int i) {
                return make_float4(wreg[4 * i], wreg[4 * i + 1], wreg[4 * i + 2], wreg[4 * i + 3]);
              });
            } else {
              const float4* wj = reinterpret_cast<const float4*>(wsm + j * 64);
              sum = weighted_head_sum(a0, a1, [&](int i) { return wj[i]; });
            }
            logit[j] = sum * scale;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[as]);
        if (c < G.ncols) {
#pragma unroll
          for (int j = 0; j < NQ; ++j) {
            if (j < G.nq) {
              const bool vis = c >= lim_lo[j] && c < lim_hi[j];
              const float v = vis ? logit[j] : ninf;
              uint32_t bits;
              if constexpr (kOutBf16) {
                const __nv_bfloat16 b = __float2bfloat16_rn(v);
                if (p.out_keep_l2) {
                  st_global_hint(reinterpret_cast<uint16_t*>(orow[j] + c), __bfloat16_as_ushort(b), pol_out);
                } else {
                  orow[j][c] = b;
                }
                bits = static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16;
              } else {
                if (p.out_keep_l2) {
                  st_global_hint(orow[j] + c, v, pol_out);
                } else {
                  orow[j][c] = v;
                }
                bits = __float_as_uint(v);
              }
              if (do_hist && vis) {
                // the key of the value as stored, so the selection sees the same digit
                const uint32_t bin = f32_key(bits) >> 22;
                atomicAdd(wh + (bin >> 1), 1u << ((bin & 1u) * 16));
              }
            }
          }
        }
        if (do_hist) {
          hist_row = G.row0;  // warp-uniform: every lane of the warp sets it
          if (++hist_tiles == 2047) flush_hist();
        }
        // next tile: the rest of this commit group, then skip the other warpgroups' groups
        ++oi;
        if ((ai + oi) % C::kCommit == 0) oi += C::kCommit * (kEpiWG - 1);
      }
      ai += nact;
      ++g;
      tb = 0;
    }
    flush_hist();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

template <int NQ, bool kOutBf16, bool kFp4 = false, bool kHist = true>
idx_status_t launch_logits(const CUtensorMap& mq, const CUtensorMap& mkv, const CUtensorMap& msc,
                           const LogitsParams& p, int grid, cudaStream_t stream, const char* fn) {
  using C = Cfg<NQ, kFp4, kHist>;
  auto kern = mqa_logits_kernel<NQ, kOutBf16, kFp4, kHist>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    // all of the unified L1 / shared memory as shared memory, so kCtasPerSm CTAs fit
    if (e == cudaSuccess) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    }
    if (e != cudaSuccess) return fail(IDX_ERR_CUDA, "%s: cudaFuncSetAttribute: %s", fn, cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(mq, mkv, msc, p);
  return check_launch(fn);
}

idx_status_t dispatch(int nq_tmpl, const CUtensorMap& mq, const CUtensorMap& mkv,
                      const CUtensorMap& msc, const LogitsParams& p, long long max_tiles,
                      cudaStream_t stream, const char* fn, bool fp4 = false) {
  const int sms = device_sm_count();
  if (sms <= 0) return fail(IDX_ERR_CUDA, "%s: cannot query the SM count", fn);
  // persistent: kCtasPerSm CTAs on every SM (fewer when there are fewer tiles)
  const int per_sm = fp4 ? Cfg<1, true>::kCtasPerSm
                         : (nq_tmpl == 1 ? Cfg<1>::kCtasPerSm
                                         : (nq_tmpl == 2 ? Cfg<2>::kCtasPerSm : Cfg<4>::kCtasPerSm));
  long long grid = static_cast<long long>(sms) * per_sm;
  if (max_tiles >= 0 && max_tiles < grid) grid = max_tiles;
  if (grid <= 0) return IDX_OK;
  // one query per group: the workspace histogram's variant (four k stages) only
  // when a workspace is given
  const int g = static_cast<int>(grid);
  const bool h = p.hist != nullptr;
  if (fp4) {
    if (nq_tmpl != 1) return fail(IDX_ERR_UNSUPPORTED, "%s: the MXFP4 path serves one query per group", fn);
    if (h) {
      return p.out_bf16 ? launch_logits<1, true, true, true>(mq, mkv, msc, p, g, stream, fn)
                        : launch_logits<1, false, true, true>(mq, mkv, msc, p, g, stream, fn);
    }
    return p.out_bf16 ? launch_logits<1, true, true, false>(mq, mkv, msc, p, g, stream, fn)
                      : launch_logits<1, false, true, false>(mq, mkv, msc, p, g, stream, fn);
  }
  switch (nq_tmpl) {
    case 1:
      if (h) {
        return p.out_bf16 ? launch_logits<1, true, false, true>(mq, mkv, msc, p, g, stream, fn)
                          : launch_logits<1, false, false, true>(mq, mkv, msc, p, g, stream, fn);
      }
      return p.out_bf16 ? launch_logits<1, true, false, false>(mq, mkv, msc, p, g, stream, fn)
                        : launch_logits<1, false, false, false>(mq, mkv, msc, p, g, stream, fn);
    case 2:
      return p.out_bf16 ? launch_logits<2, true>(mq, mkv, msc, p, static_cast<int>(grid), stream, fn)
                        : launch_logits<2, false>(mq, mkv, msc, p, static_cast<int>(grid), stream, fn);
    case 4:
      return p.out_bf16 ? launch_logits<4, true>(mq, mkv, msc, p, static_cast<int>(grid), stream, fn)
                        : launch_logits<4, false>(mq, mkv, msc, p, static_cast<int>(grid), stream, fn);
  }
  return fail(IDX_ERR_UNSUPPORTED, "%s: rows per group %d", fn, nq_tmpl);
}

idx_status_t make_q_map(CUtensorMap* m, const uint8_t* q, int64_t ld_q, int rows, int nq_box) {
  const uint64_t dims[3] = {static_cast<uint64_t>(kDim), static_cast<uint64_t>(kHeads),
                            static_cast<uint64_t>(rows)};
  const uint64_t strides[2] = {static_cast<uint64_t>(kDim), static_cast<uint64_t>(ld_q)};
  const uint32_t box[3] = {static_cast<uint32_t>(kDim), static_cast<uint32_t>(kHeads),
                           static_cast<uint32_t>(nq_box)};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, q, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

idx_status_t check_common(const char* fn, const uint8_t* q, int64_t ld_q, const void* w,
                          int w_dtype, int64_t ld_w, int rows, void* out, int out_dtype,
                          int64_t ld_out) {
  if (!q || !w || !out) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (w_dtype != IDX_F32 && w_dtype != IDX_BF16) return fail(IDX_ERR_UNSUPPORTED, "%s: w_dtype %d", fn, w_dtype);
  if (out_dtype != IDX_F32 && out_dtype != IDX_BF16) return fail(IDX_ERR_UNSUPPORTED, "%s: out_dtype %d", fn, out_dtype);
  if (ld_w < kHeads) return fail(IDX_ERR_INVALID_ARG, "%s: ld_w < 64", fn);
  if (ld_q < kHeads * kDim) return fail(IDX_ERR_INVALID_ARG, "%s: ld_q < 8192 bytes", fn);
  if (ld_q % 16 != 0 || !aligned(q, 16)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: q must be 16-byte aligned with ld_q a multiple of 16", fn);
  }
  if (rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: negative row count", fn);
  (void)ld_out;
  return IDX_OK;
}

// The optional workspace receives, per output row, the histogram of the top 10
// bits of the order-preserving key of every visible logit (the first digit of
// the selection); it must be zero on entry. Kernels with one query per group
// accumulate it.
idx_status_t attach_histogram(const char* fn, LogitsParams* p, int nq_tmpl, int rows, void* ws,
                              size_t ws_bytes) {
  if (!ws) return IDX_OK;
  if (nq_tmpl != 1) {
    return fail(IDX_ERR_UNSUPPORTED,
                "%s: the histogram workspace needs one query per group (next_n 1 or sparse mode)", fn);
  }
  const size_t need = static_cast<size_t>(rows) * kHistBins * sizeof(uint32_t);
  if (ws_bytes < need) {
    return fail(IDX_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes, need);
  }
  if (!aligned(ws, 16)) return fail(IDX_ERR_UNSUPPORTED, "%s: workspace must be 16-byte aligned", fn);
  p->hist = static_cast<uint32_t*>(ws);
  return IDX_OK;
}

bool sbk_ok(int32_t sbk) { return sbk == 8 || sbk == 16 || sbk == 32 || sbk == 64 || sbk == 128; }

}  // namespace

unsigned int logits_read_and_clear_error(cudaStream_t stream, cudaError_t* err, long long* info) {
  unsigned int v = 0;
  const unsigned int zero = 0;
  *err = cudaStreamSynchronize(stream);
  if (*err != cudaSuccess) return 0;
  *err = cudaMemcpyFromSymbol(&v, g_logits_error, sizeof(v));
  if (*err != cudaSuccess) return 0;
  if (v) {
    *err = cudaMemcpyFromSymbol(info, g_logits_error_info, 8 * sizeof(long long));
    if (*err != cudaSuccess) return v;
    *err = cudaMemcpyToSymbol(g_logits_error, &zero, sizeof(zero));
    if (*err != cudaSuccess) return v;
    *err = cudaMemcpyToSymbol(g_logits_error_taken, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace idx

using namespace idx;

namespace {

// Scores that fill at most half of L2 are stored to stay there for the
// selection that reads them next; larger ones (prefill chunks) are stored plainly.
int keep_scores_in_l2(int64_t rows, int64_t ld_out, int out_dtype) {
  const int64_t bytes = rows * ld_out * (out_dtype == IDX_BF16 ? 2 : 4);
  const int64_t l2 = device_l2_bytes();
  return l2 > 0 && bytes <= l2 / 2 ? 1 : 0;
}

// Both paged decode entry points: the e4m3 cache (132 bytes per token, fp32
// token scale) and the MXFP4 cache (68 bytes per token, E8M0 block scales).
idx_status_t paged_decode(const char* fn, bool fp4, const uint8_t* q, int64_t ld_q, const void* w,
                          int w_dtype, int64_t ld_w, const uint8_t* cache, int32_t num_blocks,
                          int32_t block_size, int64_t block_stride_bytes, const int32_t* block_table,
                          int64_t ld_bt, const int32_t* ctx_lens, int32_t B, int32_t next_n,
                          const int32_t* sparse_idx, int64_t ld_si, int32_t n_si, const int32_t* end,
                          int32_t sbk, void* logits, int out_dtype, int64_t ld_out, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
  if (B < 0 || next_n < 1) return fail(IDX_ERR_INVALID_ARG, "%s: B < 0 or next_n < 1", fn);
  if (B == 0) return IDX_OK;
  const int64_t rows64 = static_cast<int64_t>(B) * next_n;
  if (rows64 > INT32_MAX) return fail(IDX_ERR_UNSUPPORTED, "%s: too many rows", fn);
  const int rows = static_cast<int>(rows64);
  idx_status_t st = check_common(fn, q, ld_q, w, w_dtype, ld_w, rows, logits, out_dtype, ld_out);
  if (st != IDX_OK) return st;
  if (!cache || !block_table || !ctx_lens) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (num_blocks < 1) return fail(IDX_ERR_INVALID_ARG, "%s: num_blocks < 1", fn);
  if (!(block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: block_size %d is not one of 16, 32, 64, 128", fn, block_size);
  }
  const int token_bytes = fp4 ? kMxTokenBytes : kTokenBytes;
  const int row_bytes = fp4 ? kDim / 2 : kDim;  // element bytes of one token
  if (block_stride_bytes < static_cast<int64_t>(block_size) * token_bytes) {
    return fail(IDX_ERR_INVALID_ARG, "%s: block_stride_bytes < block_size * %d", fn, token_bytes);
  }
  // the FP4 tensor map reads 32-byte aligned packed rows
  const int align = fp4 ? 32 : 16;
  if (block_stride_bytes % align != 0 || !aligned(cache, align)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: cache must be %d-byte aligned with a stride multiple of %d", fn,
                align, align);
  }
  if (ld_bt < 1) return fail(IDX_ERR_INVALID_ARG, "%s: ld_bt < 1", fn);

  LogitsParams p{};
  p.n_rows = rows;
  p.next_n = next_n;
  p.w = w;
  p.w_bf16 = w_dtype == IDX_BF16;
  p.ld_w = ld_w;
  p.paged = 1;
  p.kv_base = cache;
  p.kv_block_stride = block_stride_bytes;
  p.block_size = block_size;
  p.block_table = block_table;
  p.ld_bt = ld_bt;
  p.ctx_lens = ctx_lens;
  p.out = logits;
  p.out_bf16 = out_dtype == IDX_BF16;
  p.ld_out = ld_out;
  p.out_keep_l2 = keep_scores_in_l2(rows, ld_out, out_dtype);
  int nq_tmpl = 1;
  long long max_tiles = -1;
  if (sparse_idx) {
    if (!end) return fail(IDX_ERR_INVALID_ARG, "%s: sparse mode needs end", fn);
    if (!sbk_ok(sbk) || block_size % sbk != 0) {
      return fail(IDX_ERR_UNSUPPORTED, "%s: sbk %d must be one of 8..128 and divide block_size %d", fn, sbk, block_size);
    }
    if (n_si < 1 || ld_si < n_si) return fail(IDX_ERR_INVALID_ARG, "%s: n_si < 1 or ld_si < n_si", fn);
    const int64_t ncols = static_cast<int64_t>(n_si) * sbk;
    if (ncols > INT32_MAX / 2) return fail(IDX_ERR_UNSUPPORTED, "%s: too many sparse columns", fn);
    if (ld_out < ncols) return fail(IDX_ERR_INVALID_ARG, "%s: ld_out < n_si * sbk", fn);
    p.mode = kDecodeSparse;
    p.n_groups = rows;
    p.tiles_per_group = static_cast<int>((ncols + kTile - 1) / kTile);
    p.unit = sbk;
    p.sparse_idx = sparse_idx;
    p.ld_si = ld_si;
    p.n_si = n_si;
    p.end = end;
    p.sbk = sbk;
    max_tiles = static_cast<long long>(p.n_groups) * p.tiles_per_group;
  } else {
    if (!(next_n == 1 || next_n == 2 || next_n == 4) || (fp4 && next_n != 1)) {
      return fail(IDX_ERR_UNSUPPORTED, "%s: dense decode supports next_n %s (got %d)", fn,
                  fp4 ? "1" : "1, 2 or 4", next_n);
    }
    p.mode = kDecodeDense;
    p.n_groups = B;
    p.nq = next_n;
    p.unit = block_size;
    nq_tmpl = next_n;
  }
  p.scale_slot = p.unit * 4 < 128 ? 128 : p.unit * 4;
  p.unit_shift = __builtin_ctz(static_cast<unsigned>(p.unit));
  p.slot_shift = __builtin_ctz(static_cast<unsigned>(p.scale_slot));
  st = attach_histogram(fn, &p, nq_tmpl, rows, ws, ws_bytes);
  if (st != IDX_OK) return st;

  CUtensorMap mq, mkv, msc;
  st = make_q_map(&mq, q, ld_q, rows, nq_tmpl);
  if (st != IDX_OK) return st;
  {
    // MXFP4: 128 four-bit elements per row (64 packed bytes) that the copy spreads
    // into 16-byte groups of 16 elements, giving the same 128-byte shared-memory
    // rows and swizzle as e4m3
    const uint64_t dims[3] = {static_cast<uint64_t>(kDim), static_cast<uint64_t>(block_size),
                              static_cast<uint64_t>(num_blocks)};
    const uint64_t strides[2] = {static_cast<uint64_t>(row_bytes), static_cast<uint64_t>(block_stride_bytes)};
    const uint32_t box[3] = {static_cast<uint32_t>(kDim), static_cast<uint32_t>(p.unit), 1u};
    st = encode_tensor_map(&mkv, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                           3, cache, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != IDX_OK) return st;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(block_size), static_cast<uint64_t>(num_blocks)};
    const uint64_t strides[1] = {static_cast<uint64_t>(block_stride_bytes)};
    const uint32_t box[2] = {static_cast<uint32_t>(p.unit), 1u};
    // one 4-byte word per token: the fp32 scale, or the four E8M0 block codes
    st = encode_tensor_map(&msc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                           cache + static_cast<int64_t>(block_size) * row_bytes, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != IDX_OK) return st;
  }
  return dispatch(nq_tmpl, mq, mkv, msc, p, max_tiles, stream, fn, fp4);
}

}  // namespace

extern "C" idx_status_t idx_paged_mqa_logits_decode(
    const uint8_t* q, int64_t ld_q, const void* w, int w_dtype, int64_t ld_w, const uint8_t* cache,
    int32_t num_blocks, int32_t block_size, int64_t block_stride_bytes, const int32_t* block_table,
    int64_t ld_bt, const int32_t* ctx_lens, int32_t B, int32_t next_n, const int32_t* sparse_idx,
    int64_t ld_si, int32_t n_si, const int32_t* end, int32_t sbk, void* logits, int out_dtype,
    int64_t ld_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return paged_decode("idx_paged_mqa_logits_decode", false, q, ld_q, w, w_dtype, ld_w, cache, num_blocks,
                      block_size, block_stride_bytes, block_table, ld_bt, ctx_lens, B, next_n, sparse_idx,
                      ld_si, n_si, end, sbk, logits, out_dtype, ld_out, ws, ws_bytes, stream);
}

extern "C" idx_status_t idx_paged_mqa_logits_decode_mxfp4(
    const uint8_t* q, int64_t ld_q, const void* w, int w_dtype, int64_t ld_w, const uint8_t* cache,
    int32_t num_blocks, int32_t block_size, int64_t block_stride_bytes, const int32_t* block_table,
    int64_t ld_bt, const int32_t* ctx_lens, int32_t B, int32_t next_n, const int32_t* sparse_idx,
    int64_t ld_si, int32_t n_si, const int32_t* end, int32_t sbk, void* logits, int out_dtype,
    int64_t ld_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return paged_decode("idx_paged_mqa_logits_decode_mxfp4", true, q, ld_q, w, w_dtype, ld_w, cache,
                      num_blocks, block_size, block_stride_bytes, block_table, ld_bt, ctx_lens, B, next_n,
                      sparse_idx, ld_si, n_si, end, sbk, logits, out_dtype, ld_out, ws, ws_bytes, stream);
}

namespace {

// Both prefill entry points: e4m3 k (k = k8 [S, 128], kscale = fp32 [S]) and
// MXFP4 k (k = packed e2m1 codes [S, 64], kscale = 32-bit words of E8M0 codes
// [S]; sparse mode only, the V4.1 path).
idx_status_t prefill(const char* fn, bool fp4, const uint8_t* q, int64_t ld_q, const void* w,
                     int w_dtype, int64_t ld_w, const uint8_t* k8, const void* kscale, int32_t S,
                     const int32_t* row_ks, const int32_t* row_ke, int32_t T, const int32_t* sparse_idx,
                     int64_t ld_si, int32_t n_si, const int32_t* end, int32_t sbk, void* logits,
                     int out_dtype, int64_t ld_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (T < 0 || S < 0) return fail(IDX_ERR_INVALID_ARG, "%s: negative T or S", fn);
  if (fp4 && !sparse_idx) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: MXFP4 k is scored in the sparse mode only", fn);
  }
  if (T == 0) return IDX_OK;
  idx_status_t st = check_common(fn, q, ld_q, w, w_dtype, ld_w, T, logits, out_dtype, ld_out);
  if (st != IDX_OK) return st;
  if (S == 0) return sparse_idx ? fail(IDX_ERR_INVALID_ARG, "%s: sparse mode with S == 0", fn) : IDX_OK;
  if (!k8 || !kscale) return fail(IDX_ERR_INVALID_ARG, "%s: NULL k or its scales", fn);
  // the four-bit tensor map reads 32-byte aligned rows
  if (!aligned(k8, fp4 ? 32 : 16) || !aligned(kscale, 16)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: k must be %d-byte and its scales 16-byte aligned", fn, fp4 ? 32 : 16);
  }
  LogitsParams p{};
  p.n_rows = T;
  p.next_n = 1;
  p.w = w;
  p.w_bf16 = w_dtype == IDX_BF16;
  p.ld_w = ld_w;
  p.paged = 0;
  p.kv_base = k8;
  p.kv_block_stride = 0;
  p.block_size = 1;
  p.S = S;
  p.row_ks = row_ks;
  p.row_ke = row_ke;
  p.out = logits;
  p.out_bf16 = out_dtype == IDX_BF16;
  p.ld_out = ld_out;
  p.out_keep_l2 = keep_scores_in_l2(T, ld_out, out_dtype);
  int nq_tmpl;
  if (sparse_idx) {
    if (!end) return fail(IDX_ERR_INVALID_ARG, "%s: sparse mode needs end", fn);
    if (!sbk_ok(sbk)) return fail(IDX_ERR_UNSUPPORTED, "%s: sbk %d is not one of 8..128", fn, sbk);
    if (n_si < 1 || ld_si < n_si) return fail(IDX_ERR_INVALID_ARG, "%s: n_si < 1 or ld_si < n_si", fn);
    const int64_t ncols = static_cast<int64_t>(n_si) * sbk;
    if (ncols > INT32_MAX / 2) return fail(IDX_ERR_UNSUPPORTED, "%s: too many sparse columns", fn);
    if (ld_out < ncols) return fail(IDX_ERR_INVALID_ARG, "%s: ld_out < n_si * sbk", fn);
    p.mode = kPrefillSparse;
    p.n_groups = T;
    p.tiles_per_group = static_cast<int>((ncols + kTile - 1) / kTile);
    p.unit = sbk;
    p.sparse_idx = sparse_idx;
    p.ld_si = ld_si;
    p.n_si = n_si;
    p.end = end;
    p.sbk = sbk;
    nq_tmpl = 1;
  } else {
    if (!row_ke) return fail(IDX_ERR_INVALID_ARG, "%s: dense mode needs row_ke", fn);
    if (ld_out < S) return fail(IDX_ERR_INVALID_ARG, "%s: ld_out < S", fn);
    p.mode = kPrefillDense;
    p.nq = 4;
    p.n_groups = (T + 3) / 4;
    p.tiles_per_group = (S + kTile - 1) / kTile;
    p.unit = kTile;
    nq_tmpl = 4;
  }
  p.scale_slot = p.unit * 4 < 128 ? 128 : p.unit * 4;
  p.unit_shift = __builtin_ctz(static_cast<unsigned>(p.unit));
  p.slot_shift = __builtin_ctz(static_cast<unsigned>(p.scale_slot));
  st = attach_histogram(fn, &p, nq_tmpl, T, ws, ws_bytes);
  if (st != IDX_OK) return st;
  CUtensorMap mq, mkv, msc;
  st = make_q_map(&mq, q, ld_q, T, nq_tmpl);
  if (st != IDX_OK) return st;
  {
    // MXFP4: 128 four-bit elements per row (64 packed bytes), spread by the copy
    // into the same 128-byte shared-memory rows and swizzle as e4m3
    const uint64_t row_bytes = fp4 ? kDim / 2 : kDim;
    const uint64_t dims[3] = {static_cast<uint64_t>(kDim), static_cast<uint64_t>(S), 1ull};
    const uint64_t strides[2] = {row_bytes, row_bytes * S};
    const uint32_t box[3] = {static_cast<uint32_t>(kDim), static_cast<uint32_t>(p.unit), 1u};
    st = encode_tensor_map(&mkv, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                           k8, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != IDX_OK) return st;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(S), 1ull};
    const uint64_t strides[1] = {(static_cast<uint64_t>(S) * 4 + 15) / 16 * 16};
    const uint32_t box[2] = {static_cast<uint32_t>(p.unit), 1u};
    st = encode_tensor_map(&msc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, kscale, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != IDX_OK) return st;
  }
  return dispatch(nq_tmpl, mq, mkv, msc, p, static_cast<long long>(p.n_groups) * p.tiles_per_group,
                  stream, fn, fp4);
}

}  // namespace

extern "C" idx_status_t idx_mqa_logits_prefill(const uint8_t* q, int64_t ld_q, const void* w,
                                               int w_dtype, int64_t ld_w, const uint8_t* k8,
                                               const float* kscale, int32_t S,
                                               const int32_t* row_ks, const int32_t* row_ke,
                                               int32_t T, const int32_t* sparse_idx, int64_t ld_si,
                                               int32_t n_si, const int32_t* end, int32_t sbk,
                                               void* logits, int out_dtype, int64_t ld_out,
                                               void* ws, size_t ws_bytes, cudaStream_t stream) {
  return prefill("idx_mqa_logits_prefill", false, q, ld_q, w, w_dtype, ld_w, k8, kscale, S, row_ks, row_ke,
                 T, sparse_idx, ld_si, n_si, end, sbk, logits, out_dtype, ld_out, ws, ws_bytes, stream);
}

extern "C" idx_status_t idx_mqa_logits_prefill_mxfp4(const uint8_t* q, int64_t ld_q, const void* w,
                                                     int w_dtype, int64_t ld_w, const uint8_t* k_codes,
                                                     const uint32_t* k_scales, int32_t S,
                                                     const int32_t* row_ks, const int32_t* row_ke,
                                                     int32_t T, const int32_t* sparse_idx, int64_t ld_si,
                                                     int32_t n_si, const int32_t* end, int32_t sbk,
                                                     void* logits, int out_dtype, int64_t ld_out,
                                                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  return prefill("idx_mqa_logits_prefill_mxfp4", true, q, ld_q, w, w_dtype, ld_w, k_codes, k_scales, S, row_ks,
                 row_ke, T, sparse_idx, ld_si, n_si, end, sbk, logits, out_dtype, ld_out, ws, ws_bytes, stream);
}
