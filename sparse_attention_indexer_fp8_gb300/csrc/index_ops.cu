// Integer index kernels of the indexer path:
//   a7  idx_expand_candidates   (V4.1 candidate-block flattening: one warp per row
//                                up to 256 expanded entries, one block per row beyond)
//   a6  idx_req_to_global_slots (request-local position -> physical slot)
#include <climits>

#include "common.cuh"

namespace idx {

namespace {

// Bit 0: a row of idx_expand_candidates had ks not a multiple of sbk.
// Bit 1: a slot of idx_req_to_global_slots did not fit in int32.
__device__ unsigned int g_index_ops_error = 0;

// Exclusive prefix sum of one flag per thread over the whole block (blockDim.x a
// multiple of 32, at most 1024); also returns the block total.
__device__ __forceinline__ int block_exclusive_count(int flag, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const unsigned ballot = __ballot_sync(0xFFFFFFFFu, flag);
  const int in_warp = __popc(ballot & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(ballot);
  __syncthreads();
  if (warp == 0) {
    int v = lane < nwarps ? warp_tot[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane < nwarps) warp_tot[lane] = incl - v;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  return warp_tot[warp] + in_warp;
}

// One block per row; blockDim.x = N, a power of two >= n_cand * R. Each thread
// expands one (candidate, sub-block) pair, the block sorts the N keys with a
// bitonic network in shared memory, first occurrences are compacted in order
// (sorted + deduplicated), and the tail is padded.
__global__ void expand_candidates_kernel(const int32_t* __restrict__ cand, int64_t ld_c,
                                         int n_cand, const int32_t* __restrict__ row_ks,
                                         const int32_t* __restrict__ row_ke, int R, int sbk,
                                         int32_t* __restrict__ sparse_idx, int64_t ld_si,
                                         int32_t* __restrict__ end) {
  extern __shared__ int32_t keys[];
  __shared__ int warp_tot[32];
  __shared__ int total;
  __shared__ int last;
  const int row = blockIdx.x;
  const int i = threadIdx.x;
  const int N = blockDim.x;
  const int width = n_cand * R;
  const int64_t ks = row_ks ? static_cast<int64_t>(row_ks[row]) : 0;
  const int64_t ke = row_ke[row];
  const bool ks_ok = ks >= 0 && (ks % sbk) == 0;
  const int64_t kv_len = ke > ks ? ke - ks : 0;
  const int64_t max_block = (kv_len + sbk - 1) / sbk;

  int key = INT_MAX;
  if (ks_ok && i < width) {
    const int c = cand[row * ld_c + i / R];
    if (c >= 0) {
      const int64_t x = static_cast<int64_t>(c) * R + (i % R);
      if (x < max_block) key = static_cast<int>(x);
    }
  }
  keys[i] = key;
  __syncthreads();
  for (int size = 2; size <= N; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int j = i ^ stride;
      if (j > i) {
        const int a = keys[i];
        const int b = keys[j];
        const bool ascending = (i & size) == 0;
        if ((a > b) == ascending) {
          keys[i] = b;
          keys[j] = a;
        }
      }
      __syncthreads();
    }
  }
  const int v = keys[i];
  const int prev = i > 0 ? keys[i - 1] : -1;
  const int first = (v != INT_MAX && v != prev) ? 1 : 0;
  const int pos = block_exclusive_count(first, warp_tot, &total);
  const int n = total;
  const int32_t base = static_cast<int32_t>(ks / sbk);
  if (first) {
    sparse_idx[row * ld_si + pos] = v + base;
    if (pos == n - 1) last = v;
  }
  __syncthreads();
  const int32_t pad = n > 0 ? last + base : base;
  for (int j = n + i; j < width; j += N) sparse_idx[row * ld_si + j] = pad;
  if (i == 0) {
    int32_t e = 0;
    if (n > 0) {
      const int64_t last_start = static_cast<int64_t>(last) * sbk + ks;
      int64_t fill = ke - last_start;
      fill = fill < 1 ? 1 : (fill > sbk ? sbk : fill);
      e = static_cast<int32_t>(static_cast<int64_t>(n - 1) * sbk + fill);
    }
    end[row] = e;
    if (!ks_ok) atomicOr(&g_index_ops_error, 1u);
  }
}

// One warp per row for rows of at most 256 expanded entries (E = 1, 2, 4 or 8
// per lane; entry i of the row is element e = i / 32 of lane i % 32). The same
// steps as expand_candidates_kernel: expand, sort ascending with a bitonic
// network (partners 32 or more apart within a lane's registers, nearer ones by
// shuffles, so no barrier), keep first occurrences in order, pad the tail.
template <int E>
__global__ void __launch_bounds__(128) expand_candidates_warp_kernel(
    const int32_t* __restrict__ cand, int64_t ld_c, int rows, int n_cand,
    const int32_t* __restrict__ row_ks, const int32_t* __restrict__ row_ke, int R, int sbk,
    int32_t* __restrict__ sparse_idx, int64_t ld_si, int32_t* __restrict__ end) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int width = n_cand * R;
  const int64_t ks = row_ks ? static_cast<int64_t>(row_ks[row]) : 0;
  const int64_t ke = row_ke[row];
  const bool ks_ok = ks >= 0 && (ks % sbk) == 0;
  const int64_t kv_len = ke > ks ? ke - ks : 0;
  const int64_t max_block = (kv_len + sbk - 1) / sbk;
  int key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = e * 32 + lane;
    key[e] = INT_MAX;
    if (ks_ok && i < width) {
      const int c = cand[row * ld_c + i / R];
      if (c >= 0) {
        const int64_t x = static_cast<int64_t>(c) * R + (i % R);
        if (x < max_block) key[e] = static_cast<int>(x);
      }
    }
  }
#pragma unroll
  for (int size = 2; size <= 32 * E; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int e2 = e ^ (stride >> 5);
          if (e < e2) {
            const bool asc = ((e * 32 + lane) & size) == 0;
            const int lo = min(key[e], key[e2]);
            const int hi = max(key[e], key[e2]);
            key[e] = asc ? lo : hi;
            key[e2] = asc ? hi : lo;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const bool asc = ((e * 32 + lane) & size) == 0;
          const int other = __shfl_xor_sync(0xFFFFFFFFu, key[e], stride);
          const bool lower = (lane & stride) == 0;
          key[e] = (lower == asc) ? min(key[e], other) : max(key[e], other);
        }
      }
    }
  }
  const int32_t base = static_cast<int32_t>(ks / sbk);
  const unsigned below = (1u << lane) - 1u;
  int n = 0;
  int last = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int up = __shfl_up_sync(0xFFFFFFFFu, key[e], 1);
    const int wrap = e > 0 ? __shfl_sync(0xFFFFFFFFu, key[e > 0 ? e - 1 : 0], 31) : -1;
    const int prev = lane > 0 ? up : wrap;
    const bool first = key[e] != INT_MAX && key[e] != prev;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, first);
    if (first) sparse_idx[row * ld_si + n + __popc(m & below)] = key[e] + base;
    if (m) last = __shfl_sync(0xFFFFFFFFu, key[e], 31 - __clz(m));
    n += __popc(m);
  }
  const int32_t pad = n > 0 ? last + base : base;
  for (int j = n + lane; j < width; j += 32) sparse_idx[row * ld_si + j] = pad;
  if (lane == 0) {
    int32_t e = 0;
    if (n > 0) {
      const int64_t last_start = static_cast<int64_t>(last) * sbk + ks;
      int64_t fill = ke - last_start;
      fill = fill < 1 ? 1 : (fill > sbk ? sbk : fill);
      e = static_cast<int32_t>(static_cast<int64_t>(n - 1) * sbk + fill);
    }
    end[row] = e;
    if (!ks_ok) atomicOr(&g_index_ops_error, 1u);
  }
}

__global__ void req_to_global_kernel(const int32_t* local, int64_t ld_l, int rows, int k,
                                     const int32_t* __restrict__ row_to_req,
                                     const int32_t* __restrict__ block_table, int64_t ld_bt,
                                     int block_size, int block_span, int32_t* slots,
                                     int64_t ld_s) {
  const int64_t n = static_cast<int64_t>(rows) * k;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = t / k;
    const int64_t i = t - r * k;
    const int32_t v = local[r * ld_l + i];
    int32_t out = -1;
    if (v >= 0) {
      const int64_t lb = v / block_size;
      if (lb < ld_bt) {
        const int64_t req = row_to_req ? __ldg(row_to_req + r) : r;
        const int64_t blk = __ldg(block_table + req * ld_bt + lb);
        const int64_t s = blk * block_span + v % block_size;
        if (s >= 0 && s <= INT32_MAX) {
          out = static_cast<int32_t>(s);
        } else {
          atomicOr(&g_index_ops_error, 2u);
        }
      }
    }
    slots[r * ld_s + i] = out;
  }
}

}  // namespace

unsigned int index_ops_read_and_clear_error(cudaStream_t stream, cudaError_t* err) {
  unsigned int v = 0;
  const unsigned int zero = 0;
  *err = cudaStreamSynchronize(stream);
  if (*err != cudaSuccess) return 0;
  *err = cudaMemcpyFromSymbol(&v, g_index_ops_error, sizeof(v));
  if (*err != cudaSuccess) return 0;
  if (v) *err = cudaMemcpyToSymbol(g_index_ops_error, &zero, sizeof(zero));
  return v;
}

}  // namespace idx

using namespace idx;

extern "C" idx_status_t idx_expand_candidates(const int32_t* cand, int64_t ld_c, int32_t rows,
                                              int32_t n_cand, const int32_t* row_ks,
                                              const int32_t* row_ke, int32_t cand_block_size,
                                              int32_t sbk, int32_t* sparse_idx, int64_t ld_si,
                                              int32_t* end, cudaStream_t stream) {
  const char* fn = "idx_expand_candidates";
  if (rows < 0 || n_cand < 1) return fail(IDX_ERR_INVALID_ARG, "%s: rows < 0 or n_cand < 1", fn);
  if (sbk < 1 || cand_block_size < sbk || cand_block_size % sbk != 0) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: sbk %d must divide cand_block_size %d", fn, sbk, cand_block_size);
  }
  const int R = cand_block_size / sbk;
  if ((R & (R - 1)) != 0) return fail(IDX_ERR_UNSUPPORTED, "%s: ratio %d is not a power of two", fn, R);
  if ((n_cand & (n_cand - 1)) != 0) return fail(IDX_ERR_UNSUPPORTED, "%s: n_cand %d is not a power of two", fn, n_cand);
  const int width = n_cand * R;
  if (width > 1024) return fail(IDX_ERR_UNSUPPORTED, "%s: n_cand * ratio = %d exceeds 1024", fn, width);
  if (ld_c < n_cand || ld_si < width) return fail(IDX_ERR_INVALID_ARG, "%s: ld_c or ld_si too small", fn);
  if (rows == 0) return IDX_OK;
  if (!cand || !row_ke || !sparse_idx || !end) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (width <= 256) {
    // one warp per row, four rows per block
    const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
    if (width <= 32) {
      expand_candidates_warp_kernel<1><<<blocks, 128, 0, stream>>>(cand, ld_c, rows, n_cand, row_ks, row_ke, R,
                                                                  sbk, sparse_idx, ld_si, end);
    } else if (width <= 64) {
      expand_candidates_warp_kernel<2><<<blocks, 128, 0, stream>>>(cand, ld_c, rows, n_cand, row_ks, row_ke, R,
                                                                  sbk, sparse_idx, ld_si, end);
    } else if (width <= 128) {
      expand_candidates_warp_kernel<4><<<blocks, 128, 0, stream>>>(cand, ld_c, rows, n_cand, row_ks, row_ke, R,
                                                                  sbk, sparse_idx, ld_si, end);
    } else {
      expand_candidates_warp_kernel<8><<<blocks, 128, 0, stream>>>(cand, ld_c, rows, n_cand, row_ks, row_ke, R,
                                                                  sbk, sparse_idx, ld_si, end);
    }
    return check_launch(fn);
  }
  int threads = 32;
  while (threads < width) threads <<= 1;
  expand_candidates_kernel<<<rows, threads, threads * sizeof(int32_t), stream>>>(
      cand, ld_c, n_cand, row_ks, row_ke, R, sbk, sparse_idx, ld_si, end);
  return check_launch(fn);
}

extern "C" idx_status_t idx_req_to_global_slots(const int32_t* local, int64_t ld_l, int32_t rows,
                                                int32_t k, const int32_t* row_to_req,
                                                const int32_t* block_table, int64_t ld_bt,
                                                int32_t block_size, int32_t block_span,
                                                int32_t* slots, int64_t ld_s, cudaStream_t stream) {
  const char* fn = "idx_req_to_global_slots";
  if (rows < 0 || k < 0) return fail(IDX_ERR_INVALID_ARG, "%s: negative size", fn);
  if (block_size < 1 || ld_bt < 1) return fail(IDX_ERR_INVALID_ARG, "%s: block_size and ld_bt must be positive", fn);
  if (block_span < block_size) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: block_span %d < block_size %d", fn, block_span, block_size);
  }
  if (ld_l < k || ld_s < k) return fail(IDX_ERR_INVALID_ARG, "%s: row stride smaller than k", fn);
  if (rows == 0 || k == 0) return IDX_OK;
  if (!local || !block_table || !slots) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  const int64_t n = static_cast<int64_t>(rows) * k;
  const int block = 256;
  int64_t blocks = (n + block - 1) / block;
  const int64_t cap = static_cast<int64_t>(device_sm_count() > 0 ? device_sm_count() : 148) * 16;
  if (blocks > cap) blocks = cap;
  req_to_global_kernel<<<static_cast<unsigned>(blocks), block, 0, stream>>>(
      local, ld_l, rows, k, row_to_req, block_table, ld_bt, block_size, block_span, slots, ld_s);
  return check_launch(fn);
}
