// a1: fused k quantisation + paged-cache insert, and the prefill gather of k.
//
// "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", "Indexer 内部六步" step 5: k is
// quantised to FP8 while it is written into the indexer cache (132 bytes per
// token: 128 e4m3 bytes and one fp32 scale, the page's cost table). One warp
// handles one token: lane l owns dims 4l..4l+3, the warp reduces |k| to amax, and
// the lane writes its four e4m3 bytes as one 32-bit store, so a token's 128-byte
// value row leaves as one coalesced 128-byte transaction.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace idx {
namespace {

constexpr int kWarpsPerBlock = 8;

template <bool kBf16>
__device__ __forceinline__ void load4(const void* k, int64_t ld_k, int tok, int lane, bool vec,
                                      float (&x)[4]) {
  if constexpr (kBf16) {
    const uint16_t* row = static_cast<const uint16_t*>(k) + static_cast<int64_t>(tok) * ld_k + 4 * lane;
    uint16_t h[4];
    if (vec) {
      uint2 v = __ldg(reinterpret_cast<const uint2*>(row));
      h[0] = v.x & 0xFFFF; h[1] = v.x >> 16; h[2] = v.y & 0xFFFF; h[3] = v.y >> 16;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __ldg(row + i);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __uint_as_float(static_cast<uint32_t>(h[i]) << 16);
  } else {
    const float* row = static_cast<const float*>(k) + static_cast<int64_t>(tok) * ld_k + 4 * lane;
    if (vec) {
      float4 v = __ldg(reinterpret_cast<const float4*>(row));
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = __ldg(row + i);
    }
  }
}

// The smallest power of two >= s (s a positive binary32 value), the UE8M0
// scale format: an exact power of two keeps its value, anything else rounds up
// to the next exponent. 0 stays 0.
__device__ __forceinline__ float ue8m0_ceil(float s) {
  const uint32_t b = __float_as_uint(s);
  if (s == 0.0f) return 0.0f;
  const uint32_t e = b >> 23;                  // biased exponent (s > 0, finite)
  if (e == 0) {                                // subnormal: the next power of two above it
    const int lz = __clz(b);                   // b < 2^23
    return __uint_as_float(1u << (31 - lz + ((b & (b - 1)) != 0)));
  }
  return (b & 0x7FFFFFu) == 0 ? s : __uint_as_float((e + 1) << 23);
}

template <bool kBf16>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
k_quant_and_cache_kernel(const void* __restrict__ k, int64_t ld_k, int n_tok, bool vec, bool ue8m0,
                         const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ cache,
                         int64_t n_slots, int block_size, int64_t block_stride) {
  const int tok = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= n_tok) return;
  const int64_t slot = __ldg(slot_mapping + tok);
  if (slot < 0 || slot >= n_slots) return;

  float x[4];
  load4<kBf16>(k, ld_k, tok, lane, vec, x);
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));

  // IEEE binary32 divisions, correctly rounded, as the scale format fixes;
  // UE8M0 then rounds the scale up to a power of two (k / scale stays <= 448)
  float scale = __fdiv_rn(amax, 448.0f);
  if (ue8m0) scale = ue8m0_ceil(scale);
  uint32_t packed = 0;
  if (scale >= 0x1p-126f) {
    const float r = __frcp_rn(scale);
    packed = e4m3x2_of_quotients(x[0], x[1], scale, r) | (e4m3x2_of_quotients(x[2], x[3], scale, r) << 16);
  } else if (scale != 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) packed |= e4m3_of_quotient_exact(x[i], scale) << (8 * i);
  }
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot - blk * block_size);
  uint8_t* base = cache + blk * block_stride;
  *reinterpret_cast<uint32_t*>(base + off * kDim + 4 * lane) = packed;
  if (lane == 0) *reinterpret_cast<float*>(base + block_size * kDim + 4 * off) = scale;
}

// MXFP4 insert (the V4.1 cache format): the OCP MX conversion per 32-dim block.
// One warp per token, lane l owns dims 4l..4l+3, so block j is lanes 8j..8j+7.
// Shared exponent floor(log2(amax)) - 2, clamped to the E8M0 range: for a
// binary32 amax with biased exponent E that is E - 129, and its E8M0 code is
// max(E - 2, 0) (E = 0 for zero or subnormal amax, which clamps to 2^-127).
// The quotient by the power of two is a multiplication by 2^(127 - code),
// exact except where it underflows to a magnitude far below the smallest e2m1
// step, which rounds to 0 either way; cvt.rn.satfinite.e2m1x2 rounds to nearest
// even and saturates to +-6. The lane's four codes leave as one 16-bit store
// (dim 2i in the low nibble), the warp's 64 bytes as one transaction, and lane
// 0 writes the four scale codes of the token as one 32-bit word.
template <bool kBf16>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
k_quant_and_cache_mxfp4_kernel(const void* __restrict__ k, int64_t ld_k, int n_tok, bool vec,
                               const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ cache,
                               int64_t n_slots, int block_size, int64_t block_stride) {
  const int tok = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= n_tok) return;
  const int64_t slot = __ldg(slot_mapping + tok);
  if (slot < 0 || slot >= n_slots) return;

  float x[4];
  load4<kBf16>(k, ld_k, tok, lane, vec, x);
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int e = static_cast<int>(__float_as_uint(amax) >> 23);   // amax >= 0
  const uint32_t code = static_cast<uint32_t>(max(e - 2, 0));   // 0..252
  const float inv = __uint_as_float((254u - code) << 23);      // 2^(127 - code), a normal float
  const uint32_t lo = __nv_cvt_float2_to_fp4x2(make_float2(x[0] * inv, x[1] * inv), __NV_E2M1, cudaRoundNearest);
  const uint32_t hi = __nv_cvt_float2_to_fp4x2(make_float2(x[2] * inv, x[3] * inv), __NV_E2M1, cudaRoundNearest);
  // the four block codes, byte j from lane 8j
  const uint32_t c0 = __shfl_sync(0xFFFFFFFFu, code, 0), c1 = __shfl_sync(0xFFFFFFFFu, code, 8);
  const uint32_t c2 = __shfl_sync(0xFFFFFFFFu, code, 16), c3 = __shfl_sync(0xFFFFFFFFu, code, 24);
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot - blk * block_size);
  uint8_t* base = cache + blk * block_stride;
  *reinterpret_cast<uint16_t*>(base + off * (kDim / 2) + 2 * lane) = static_cast<uint16_t>(lo | (hi << 8));
  if (lane == 0) {
    *reinterpret_cast<uint32_t*>(base + block_size * (kDim / 2) + 4 * off) = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
  }
}

// One thread per 16-byte chunk: eight threads move one token's value row.
__global__ void gather_k_kernel(const uint8_t* __restrict__ cache, int block_size,
                                int64_t block_stride, const int32_t* __restrict__ block_table,
                                int n_tok, uint8_t* __restrict__ k8_out,
                                float* __restrict__ kscale_out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t p = i >> 3;
  const int chunk = static_cast<int>(i & 7);
  if (p >= n_tok) return;
  const int64_t blk = __ldg(block_table + p / block_size);
  const int off = static_cast<int>(p % block_size);
  const uint8_t* src = cache + blk * block_stride;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + off * kDim + chunk * 16));
  *reinterpret_cast<uint4*>(k8_out + p * kDim + chunk * 16) = v;
  if (chunk == 0) {
    kscale_out[p] = __ldg(reinterpret_cast<const float*>(src + block_size * kDim + 4 * off));
  }
}

// The MXFP4 twin: one thread per 16-byte chunk, four threads move one token's
// 64 bytes of e2m1 codes and the first also moves its word of E8M0 scale codes.
__global__ void gather_k_mxfp4_kernel(const uint8_t* __restrict__ cache, int block_size,
                                      int64_t block_stride, const int32_t* __restrict__ block_table,
                                      int n_tok, uint8_t* __restrict__ codes_out,
                                      uint32_t* __restrict__ scales_out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t p = i >> 2;
  const int chunk = static_cast<int>(i & 3);
  if (p >= n_tok) return;
  const int64_t blk = __ldg(block_table + p / block_size);
  const int off = static_cast<int>(p % block_size);
  const uint8_t* src = cache + blk * block_stride;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + off * (kDim / 2) + chunk * 16));
  *reinterpret_cast<uint4*>(codes_out + p * (kDim / 2) + chunk * 16) = v;
  if (chunk == 0) {
    scales_out[p] = __ldg(reinterpret_cast<const uint32_t*>(src + block_size * (kDim / 2) + 4 * off));
  }
}

bool block_size_ok(int32_t bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128; }

idx_status_t check_cache(const char* fn, const void* cache, int32_t block_size,
                         int64_t block_stride) {
  if (!block_size_ok(block_size)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: block_size %d is not one of 16, 32, 64, 128", fn, block_size);
  }
  if (block_stride < static_cast<int64_t>(block_size) * kTokenBytes) {
    return fail(IDX_ERR_INVALID_ARG, "%s: block_stride_bytes %lld < block_size * 132", fn,
                static_cast<long long>(block_stride));
  }
  if (block_stride % 16 != 0) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: block_stride_bytes %lld is not a multiple of 16", fn,
                static_cast<long long>(block_stride));
  }
  if (!aligned(cache, 16)) return fail(IDX_ERR_UNSUPPORTED, "%s: cache is not 16-byte aligned", fn);
  return IDX_OK;
}

idx_status_t check_cache_mxfp4(const char* fn, const void* cache, int32_t block_size,
                               int64_t block_stride) {
  if (!block_size_ok(block_size)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: block_size %d is not one of 16, 32, 64, 128", fn, block_size);
  }
  if (block_stride < static_cast<int64_t>(block_size) * IDX_MXFP4_TOKEN_BYTES) {
    return fail(IDX_ERR_INVALID_ARG, "%s: block_stride_bytes %lld < block_size * 68", fn,
                static_cast<long long>(block_stride));
  }
  if (block_stride % 32 != 0) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: block_stride_bytes %lld is not a multiple of 32", fn,
                static_cast<long long>(block_stride));
  }
  if (!aligned(cache, 32)) return fail(IDX_ERR_UNSUPPORTED, "%s: cache is not 32-byte aligned", fn);
  return IDX_OK;
}

}  // namespace
}  // namespace idx

using namespace idx;

extern "C" idx_status_t idx_k_quant_and_cache(const void* k, int k_dtype, int64_t ld_k,
                                              int32_t n_tok, const int64_t* slot_mapping,
                                              uint8_t* cache, int32_t num_blocks,
                                              int32_t block_size, int64_t block_stride_bytes,
                                              int scale_fmt, cudaStream_t stream) {
  const char* fn = "idx_k_quant_and_cache";
  if (n_tok < 0 || num_blocks < 0) return fail(IDX_ERR_INVALID_ARG, "%s: negative size", fn);
  if (k_dtype != IDX_BF16 && k_dtype != IDX_F32) return fail(IDX_ERR_UNSUPPORTED, "%s: k_dtype %d", fn, k_dtype);
  if (scale_fmt != IDX_SCALE_FP32 && scale_fmt != IDX_SCALE_UE8M0) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: scale_fmt %d", fn, scale_fmt);
  }
  if (ld_k < kDim) return fail(IDX_ERR_INVALID_ARG, "%s: ld_k %lld < 128", fn, static_cast<long long>(ld_k));
  if (n_tok == 0) return IDX_OK;
  if (!k || !slot_mapping || !cache) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  idx_status_t st = check_cache(fn, cache, block_size, block_stride_bytes);
  if (st != IDX_OK) return st;
  const size_t esz = k_dtype == IDX_BF16 ? 2 : 4;
  const size_t vec_bytes = 4 * esz;
  const bool vec = aligned(k, vec_bytes) && (static_cast<size_t>(ld_k) * esz) % vec_bytes == 0;
  const int64_t n_slots = static_cast<int64_t>(num_blocks) * block_size;
  const dim3 grid((n_tok + kWarpsPerBlock - 1) / kWarpsPerBlock);
  if (k_dtype == IDX_BF16) {
    k_quant_and_cache_kernel<true><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        k, ld_k, n_tok, vec, scale_fmt == IDX_SCALE_UE8M0, slot_mapping, cache, n_slots, block_size,
        block_stride_bytes);
  } else {
    k_quant_and_cache_kernel<false><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        k, ld_k, n_tok, vec, scale_fmt == IDX_SCALE_UE8M0, slot_mapping, cache, n_slots, block_size,
        block_stride_bytes);
  }
  return check_launch(fn);
}

extern "C" idx_status_t idx_gather_k(const uint8_t* cache, int32_t block_size,
                                     int64_t block_stride_bytes, const int32_t* block_table,
                                     int32_t n_tok, uint8_t* k8_out, float* kscale_out,
                                     cudaStream_t stream) {
  const char* fn = "idx_gather_k";
  if (n_tok < 0) return fail(IDX_ERR_INVALID_ARG, "%s: negative n_tok", fn);
  if (n_tok == 0) return IDX_OK;
  if (!cache || !block_table || !k8_out || !kscale_out) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  idx_status_t st = check_cache(fn, cache, block_size, block_stride_bytes);
  if (st != IDX_OK) return st;
  if (!aligned(k8_out, 16) || !aligned(kscale_out, 4)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: k8_out must be 16-byte and kscale_out 4-byte aligned", fn);
  }
  const int64_t threads = static_cast<int64_t>(n_tok) * 8;
  const int block = 256;
  const dim3 grid(static_cast<unsigned>((threads + block - 1) / block));
  gather_k_kernel<<<grid, block, 0, stream>>>(cache, block_size, block_stride_bytes, block_table,
                                              n_tok, k8_out, kscale_out);
  return check_launch(fn);
}

extern "C" idx_status_t idx_gather_k_mxfp4(const uint8_t* cache, int32_t block_size,
                                           int64_t block_stride_bytes, const int32_t* block_table,
                                           int32_t n_tok, uint8_t* codes_out, uint32_t* scales_out,
                                           cudaStream_t stream) {
  const char* fn = "idx_gather_k_mxfp4";
  if (n_tok < 0) return fail(IDX_ERR_INVALID_ARG, "%s: negative n_tok", fn);
  if (n_tok == 0) return IDX_OK;
  if (!cache || !block_table || !codes_out || !scales_out) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  idx_status_t st = check_cache_mxfp4(fn, cache, block_size, block_stride_bytes);
  if (st != IDX_OK) return st;
  if (!aligned(codes_out, 16) || !aligned(scales_out, 4)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: codes_out must be 16-byte and scales_out 4-byte aligned", fn);
  }
  const int64_t threads = static_cast<int64_t>(n_tok) * 4;
  const int block = 256;
  const dim3 grid(static_cast<unsigned>((threads + block - 1) / block));
  gather_k_mxfp4_kernel<<<grid, block, 0, stream>>>(cache, block_size, block_stride_bytes, block_table,
                                                    n_tok, codes_out, scales_out);
  return check_launch(fn);
}

extern "C" idx_status_t idx_k_quant_and_cache_mxfp4(const void* k, int k_dtype, int64_t ld_k,
                                                    int32_t n_tok, const int64_t* slot_mapping,
                                                    uint8_t* cache, int32_t num_blocks,
                                                    int32_t block_size, int64_t block_stride_bytes,
                                                    cudaStream_t stream) {
  const char* fn = "idx_k_quant_and_cache_mxfp4";
  if (n_tok < 0 || num_blocks < 0) return fail(IDX_ERR_INVALID_ARG, "%s: negative size", fn);
  if (k_dtype != IDX_BF16 && k_dtype != IDX_F32) return fail(IDX_ERR_UNSUPPORTED, "%s: k_dtype %d", fn, k_dtype);
  if (ld_k < kDim) return fail(IDX_ERR_INVALID_ARG, "%s: ld_k %lld < 128", fn, static_cast<long long>(ld_k));
  if (n_tok == 0) return IDX_OK;
  if (!k || !slot_mapping || !cache) return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  idx_status_t st = check_cache_mxfp4(fn, cache, block_size, block_stride_bytes);
  if (st != IDX_OK) return st;
  const size_t esz = k_dtype == IDX_BF16 ? 2 : 4;
  const size_t vec_bytes = 4 * esz;
  const bool vec = aligned(k, vec_bytes) && (static_cast<size_t>(ld_k) * esz) % vec_bytes == 0;
  const int64_t n_slots = static_cast<int64_t>(num_blocks) * block_size;
  const dim3 grid((n_tok + kWarpsPerBlock - 1) / kWarpsPerBlock);
  if (k_dtype == IDX_BF16) {
    k_quant_and_cache_mxfp4_kernel<true><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        k, ld_k, n_tok, vec, slot_mapping, cache, n_slots, block_size, block_stride_bytes);
  } else {
    k_quant_and_cache_mxfp4_kernel<false><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        k, ld_k, n_tok, vec, slot_mapping, cache, n_slots, block_size, block_stride_bytes);
  }
  return check_launch(fn);
}
