// Indexer q preparation: partial RoPE, per-head FP8 quantisation and the
// folding of every q-side coefficient into the head weights, in one pass.
//
// "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", "Indexer 内部六步" steps 3-4: RoPE is
// applied to the first 64 of the 128 dims only; q is quantised to FP8 with one
// scale per 128 values (one per head), and the weights absorb
// q_scale * softmax_scale * n_head_scale so the scoring kernel multiplies by no
// other coefficient; on CUDA the two steps are one fused kernel. "V4.1 索引器接入
// 稀疏 MQA logits", 实现拆解 item 5: the fused kernel can write the weights
// directly as bf16 (the fp32 value rounded once).
//
// One block per token, one warp per group of 8 heads. A warp works on two heads
// at a time, 16 lanes each, and every lane reads its 8 dims as two runs of 4
// (8-byte bf16 / 16-byte fp32 loads) chosen so that each rotary pair lies in
// one lane: for NeoX pairs (i, i + 32) lane l < 8 reads dims 4l..4l+3 and
// 32+4l..32+4l+3, for interleaved pairs (2i, 2i + 1) dims 8l..8l+7; lanes 8-15
// read the pass-through dims 64 + 8(l-8)..+7. Both styles give lane l the
// pairs 4l..4l+3. All four passes' loads are issued before any arithmetic. The
// 16 lanes reduce |q| to amax, every lane writes its two runs of e4m3 bytes in
// place, and the first lane of the half writes the folded weight.
//
// Arithmetic (IEEE binary32, each operation rounded, no contraction, so the
// bytes are reproducible): y1 = x1 c - x2 s, y2 = x2 c + x1 s;
// scale = amax / 448; q8 = e4m3_rn_satfinite(y / scale);
// w_out = ((w * scale) * softmax_scale) * n_head_scale.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace idx {

namespace {

constexpr int kWarpsPerBlock = 8;   // 8 warps x 8 heads = one token
constexpr int kPasses = 4;          // two heads per pass

// Bit 0: a position outside [0, max_pos) (the head is written as zeros).
__device__ unsigned int g_q_rope_error = 0;

struct QRopeParams {
  const void* q;
  int q_bf16;
  int64_t ld_q;  // elements between tokens
  const int32_t* positions;
  const float* cos_sin;  // [max_pos, ld_cs]: cos of the 32 pair angles, then their sin
  int64_t ld_cs;
  int max_pos;
  int interleaved;
  const void* w;
  int w_bf16;
  int64_t ld_w;
  float softmax_scale;
  float n_head_scale;
  int T;
  uint8_t* q8;
  int64_t ld_q8;  // bytes between tokens
  void* w_out;
  int w_out_bf16;
  int64_t ld_wo;
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Four consecutive q values at element offset `off` of the row.
__device__ __forceinline__ void load_run(const QRopeParams& p, int64_t off, float* v) {
  if (p.q_bf16) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.q) + off));
    v[0] = bf16_bits_to_float(u.x & 0xFFFF);
    v[1] = bf16_bits_to_float(u.x >> 16);
    v[2] = bf16_bits_to_float(u.y & 0xFFFF);
    v[3] = bf16_bits_to_float(u.y >> 16);
  } else {
    const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.q) + off));
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  }
}

template <bool kInterleaved>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) q_rope_quant_kernel(const QRopeParams p) {
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;        // lane within the head's half-warp
  const int half = lane >> 4;      // which of the pass's two heads
  const bool rot = hl < 8;
  // element offsets (within a head) of this lane's two runs of four dims
  const int off0 = rot ? (kInterleaved ? 8 * hl : 4 * hl) : 64 + 8 * (hl - 8);
  const int off1 = rot ? (kInterleaved ? 8 * hl + 4 : 32 + 4 * hl) : 64 + 8 * (hl - 8) + 4;

  float raw[kPasses][8];
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int h = 8 * warp + 2 * ps + half;
    const int64_t base = static_cast<int64_t>(t) * p.ld_q + h * kDim;
    load_run(p, base + off0, raw[ps]);
    load_run(p, base + off1, raw[ps] + 4);
  }

  int pos = __ldg(p.positions + t);
  const bool pos_ok = pos >= 0 && pos < p.max_pos;
  if (!pos_ok) {
    if (threadIdx.x == 0) atomicOr(&g_q_rope_error, 1u);
    pos = 0;
  }
  float4 c4 = make_float4(1.f, 1.f, 1.f, 1.f), s4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (rot) {  // cos / sin of pairs 4hl..4hl+3
    const float* cs = p.cos_sin + static_cast<int64_t>(pos) * p.ld_cs + 4 * hl;
    c4 = __ldg(reinterpret_cast<const float4*>(cs));
    s4 = __ldg(reinterpret_cast<const float4*>(cs + 32));
  }
  const float c[4] = {c4.x, c4.y, c4.z, c4.w};
  const float sn[4] = {s4.x, s4.y, s4.z, s4.w};

#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int h = 8 * warp + 2 * ps + half;
    const float* r = raw[ps];
    float v[8];  // the lane's dims in load order: run 0, then run 1
    if (rot) {
      // pair i of the lane: members (a, b) = (r[i], r[4 + i]) for NeoX,
      // (r[2i], r[2i + 1]) for interleaved (runs 8hl..8hl+3, 8hl+4..8hl+7)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ia = kInterleaved ? 2 * i : i;
        const int ib = kInterleaved ? 2 * i + 1 : 4 + i;
        const float a = r[ia], b = r[ib];
        v[ia] = __fsub_rn(__fmul_rn(a, c[i]), __fmul_rn(b, sn[i]));
        v[ib] = __fadd_rn(__fmul_rn(b, c[i]), __fmul_rn(a, sn[i]));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = r[i];
    }
    if (!pos_ok) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }

    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float scale = __fdiv_rn(amax, 448.0f);
    uint32_t packed[2] = {0u, 0u};
    if (scale >= 0x1p-126f) {
      const float rs = __frcp_rn(scale);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        packed[i >> 2] |= e4m3x2_of_quotients(v[i], v[i + 1], scale, rs) << (8 * (i & 3));
      }
    } else if (scale != 0.0f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) packed[i >> 2] |= e4m3_of_quotient_exact(v[i], scale) << (8 * (i & 3));
    }
    uint8_t* dst = p.q8 + static_cast<int64_t>(t) * p.ld_q8 + h * kDim;
    *reinterpret_cast<uint32_t*>(dst + off0) = packed[0];
    *reinterpret_cast<uint32_t*>(dst + off1) = packed[1];

    if (hl == 0) {
      const int64_t wi = static_cast<int64_t>(t) * p.ld_w + h;
      const float w = p.w_bf16 ? bf16_bits_to_float(__ldg(static_cast<const uint16_t*>(p.w) + wi))
                               : __ldg(static_cast<const float*>(p.w) + wi);
      const float wf = __fmul_rn(__fmul_rn(__fmul_rn(w, scale), p.softmax_scale), p.n_head_scale);
      const int64_t wo = static_cast<int64_t>(t) * p.ld_wo + h;
      if (p.w_out_bf16) {
        static_cast<__nv_bfloat16*>(p.w_out)[wo] = __float2bfloat16_rn(wf);
      } else {
        static_cast<float*>(p.w_out)[wo] = wf;
      }
    }
  }
}

}  // namespace

unsigned int q_rope_read_and_clear_error(cudaStream_t stream, cudaError_t* err) {
  unsigned int v = 0;
  const unsigned int zero = 0;
  *err = cudaStreamSynchronize(stream);
  if (*err != cudaSuccess) return 0;
  *err = cudaMemcpyFromSymbol(&v, g_q_rope_error, sizeof(v));
  if (*err != cudaSuccess) return 0;
  if (v) *err = cudaMemcpyToSymbol(g_q_rope_error, &zero, sizeof(zero));
  return v;
}

}  // namespace idx

using namespace idx;

extern "C" idx_status_t idx_q_rope_quant(const void* q, int q_dtype, int64_t ld_q,
                                         const int32_t* positions, const float* cos_sin,
                                         int64_t ld_cs, int32_t max_pos, int32_t rope_style,
                                         const void* w, int w_dtype, int64_t ld_w,
                                         float softmax_scale, float n_head_scale, int32_t T,
                                         uint8_t* q8, int64_t ld_q8, void* w_out, int w_out_dtype,
                                         int64_t ld_wo, cudaStream_t stream) {
  const char* fn = "idx_q_rope_quant";
  if (T < 0 || max_pos < 1) return fail(IDX_ERR_INVALID_ARG, "%s: T < 0 or max_pos < 1", fn);
  if ((q_dtype != IDX_F32 && q_dtype != IDX_BF16) || (w_dtype != IDX_F32 && w_dtype != IDX_BF16) ||
      (w_out_dtype != IDX_F32 && w_out_dtype != IDX_BF16)) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: element types must be IDX_F32 or IDX_BF16", fn);
  }
  if (rope_style != IDX_ROPE_NEOX && rope_style != IDX_ROPE_INTERLEAVED) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: rope_style %d", fn, rope_style);
  }
  if (ld_q < kHeads * kDim || ld_q8 < kHeads * kDim || ld_w < kHeads || ld_wo < kHeads || ld_cs < 64) {
    return fail(IDX_ERR_INVALID_ARG, "%s: a stride is smaller than its row", fn);
  }
  if (T == 0) return IDX_OK;
  if (!q || !positions || !cos_sin || !w || !q8 || !w_out) {
    return fail(IDX_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  }
  const int esz = q_dtype == IDX_BF16 ? 2 : 4;
  if (!aligned(q, 16) || (ld_q * esz) % 16 != 0) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: q rows must be 16-byte aligned", fn);
  }
  if (!aligned(q8, 16) || ld_q8 % 16 != 0) {
    return fail(IDX_ERR_UNSUPPORTED, "%s: q8 rows must be 16-byte aligned", fn);
  }
  QRopeParams p{};
  p.q = q;
  p.q_bf16 = q_dtype == IDX_BF16;
  p.ld_q = ld_q;
  p.positions = positions;
  p.cos_sin = cos_sin;
  p.ld_cs = ld_cs;
  p.max_pos = max_pos;
  p.interleaved = rope_style == IDX_ROPE_INTERLEAVED;
  p.w = w;
  p.w_bf16 = w_dtype == IDX_BF16;
  p.ld_w = ld_w;
  p.softmax_scale = softmax_scale;
  p.n_head_scale = n_head_scale;
  p.T = T;
  p.q8 = q8;
  p.ld_q8 = ld_q8;
  p.w_out = w_out;
  p.w_out_bf16 = w_out_dtype == IDX_BF16;
  p.ld_wo = ld_wo;
  static_assert(kWarpsPerBlock * kPasses * 2 == kHeads, "one block per token");
  if (p.interleaved) {
    q_rope_quant_kernel<true><<<static_cast<unsigned>(T), kWarpsPerBlock * 32, 0, stream>>>(p);
  } else {
    q_rope_quant_kernel<false><<<static_cast<unsigned>(T), kWarpsPerBlock * 32, 0, stream>>>(p);
  }
  return check_launch(fn);
}
