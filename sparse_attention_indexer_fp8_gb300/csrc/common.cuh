// Shared host and device helpers of libidx: status reporting, device queries and
// the thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and the
// 5th-generation tensor core (tcgen05) that the kernels are written against.
#pragma once

#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "idx.h"

namespace idx {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kTokenBytes = 132;
constexpr int kMxTokenBytes = 68;  // MXFP4 cache: 64 bytes of e2m1 elements + 4 E8M0 scale codes

// ---------------------------------------------------------------------------
// host-side status helpers (defined in api.cu)
// ---------------------------------------------------------------------------
idx_status_t fail(idx_status_t st, const char* fmt, ...);
idx_status_t check_launch(const char* what);
int device_sm_count();
int64_t device_l2_bytes();  // 0 when it cannot be queried
// True when a selection over `rows` rows of at most `max_cols` columns runs the
// short-row kernel, which does not read the first-digit histogram (defined in topk.cu).
bool topk_rows_short(int64_t rows, int64_t max_cols);

// Encodes a tiled TMA descriptor through the driver entry point (no -lcuda link).
idx_status_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank,
                               const void* base, const uint64_t* dims,
                               const uint64_t* strides_bytes, const uint32_t* box,
                               CUtensorMapSwizzle swizzle);

// Per-translation-unit readers of device error flags, registered in api.cu.
unsigned int logits_read_and_clear_error(cudaStream_t stream, cudaError_t* err, long long* info);
unsigned int index_ops_read_and_clear_error(cudaStream_t stream, cudaError_t* err);
unsigned int q_rope_read_and_clear_error(cudaStream_t stream, cudaError_t* err);
unsigned int topk_read_and_clear_error(cudaStream_t stream, cudaError_t* err);
unsigned int diag_read_and_clear_error(cudaStream_t stream, cudaError_t* err);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Order-preserving map of an fp32 bit pattern onto uint32 (larger value -> larger key).
__device__ __forceinline__ uint32_t f32_key(uint32_t u) {
  // negative: all bits flipped; positive: the sign bit set
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// --- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// --- TMA ---------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Global stores that carry an L2 eviction policy (an earlier createpolicy).
__device__ __forceinline__ void st_global_hint(float* ptr, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(pol) : "memory");
}

__device__ __forceinline__ void st_global_hint(uint16_t* ptr, uint16_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(ptr), "h"(v), "l"(pol) : "memory");
}

// Asks the memory system to bring [ptr, ptr + bytes) into L2 (a bulk
// asynchronous prefetch: no destination, nothing to wait for). ptr 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}

// --- e4m3 quantisation ----------------------------------------------------------
// e4m3 codes (round to nearest even, saturating to 448) of fl32(x0 / s) and
// fl32(x1 / s), x0 in the low byte, where fl32 is the correctly rounded
// binary32 quotient; r must be fl32(1 / s) (__frcp_rn) and s a positive normal.
//
// q = fl32(x * r) lies within 1.5 * 2^-23 (relative) of x / s, and fl32(x / s)
// within a further 2^-24, so both lie strictly inside [q (1 - 2^-21), q (1 + 2^-21)]
// (the two bounds, rounded to binary32, are still at least 3.5 ulps away from q).
// The conversion is monotonic: when both bounds convert to the same code, so
// does fl32(x / s). Otherwise q is within a few ulps of a rounding boundary and
// the quotient is computed exactly. This keeps the bytes identical to the
// division-per-element definition at a fraction of its cost.
__device__ __forceinline__ uint32_t e4m3x2_of_quotients(float x0, float x1, float s, float r) {
  constexpr float kUp = 1.0f + 0x1p-21f;
  constexpr float kDown = 1.0f - 0x1p-21f;
  const float q0 = __fmul_rn(x0, r);
  const float q1 = __fmul_rn(x1, r);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(q0, kUp), __fmul_rn(q1, kUp)),
                                               __NV_SATFINITE, __NV_E4M3);
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(q0, kDown), __fmul_rn(q1, kDown)),
                                               __NV_SATFINITE, __NV_E4M3);
  if (hi == lo) return hi;
  const uint32_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(x0, s), __NV_SATFINITE, __NV_E4M3);
  const uint32_t c1 = __nv_cvt_float_to_fp8(__fdiv_rn(x1, s), __NV_SATFINITE, __NV_E4M3);
  return c0 | (c1 << 8);
}

// e4m3 code of fl32(x / s) by the division itself (any positive s).
__device__ __forceinline__ uint32_t e4m3_of_quotient_exact(float x, float s) {
  return __nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3);
}

// --- tcgen05 -----------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand staged by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked
// along M/N (stride byte offset 1024). Fields: start address >> 4 in bits 0-13,
// leading byte offset >> 4 in bits 16-29 (unused for swizzled K-major),
// stride byte offset >> 4 in bits 32-45, the fixed value 1 in bits 46-47,
// swizzle mode 2 (128-byte) in bits 61-63.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with e4m3 A and B, fp32
// accumulation, both operands K-major: D format in bits 4-5 (1 = f32), A/B
// formats in bits 7-9 / 10-12 (0 = e4m3), N >> 3 in bits 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of the block-scaled tcgen05.mma kind::mxf8f6f4 with FP4
// e2m1 A (k) and e4m3 B (q), fp32 accumulation, both operands K-major: B's
// scale-factor id in bits 4-5, A/B formats in bits 7-9 / 10-12 (e2m1 = 5,
// e4m3 = 0), N >> 3 in bits 17-22, scale type UE8M0 (1) in bit 23, M >> 4 in
// bits 24-28, A's scale-factor id in bits 29-30. The ids pick the byte of each
// 32-bit scale word that the instruction's K block (32 elements) uses.
__host__ __device__ constexpr uint32_t idesc_mx_e2m1_e4m3(int M, int N) {
  return (5u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t idesc_with_scale_ids(uint32_t idesc, uint32_t a_id, uint32_t b_id) {
  return idesc | (b_id << 4) | (a_id << 29);
}

// D += (A * scale_A) x (B * scale_B)^T over one K block of 32, scale_vec::1X: one
// E8M0 scale per row and K block. For M = 128 the scale of A's row r is read
// from tensor-memory lane r, column sfa + r / 32 (byte = the A id); B's from
// sfb likewise.
__device__ __forceinline__ void umma_mx_e2m1_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                  uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads of them (a tensor-memory copy or an MMA operand).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory descriptor of 32 consecutive 16-byte lines (no swizzle: 8-line
// core matrices of 128 bytes, the next one 128 bytes on), the source of a
// tcgen05.cp of shape 32x128b. Fields as in sw128_kmajor_desc, swizzle mode 0.
__device__ __forceinline__ uint64_t lines_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 16;
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Copies 32 lines of 16 bytes from shared memory into tensor memory, line m into
// lane m of each of the four lane quarters, four 32-bit columns from taddr.
// Asynchronous, in issue order with this thread's later tcgen05.mma.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t src_desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc) : "memory");
}

// Each thread of the warp writes 32-bit words to its own TMEM lane: one column,
// or four consecutive columns. Complete with tmem_wait_st() before signalling.
__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0),
               "r"(v1), "r"(v2), "r"(v3)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Each thread of the warp reads 32 consecutive fp32 columns of its own TMEM lane.
// The values are only valid after tmem_wait_ld(), which takes them as operands so
// the compiler cannot consume them before the wait.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// Orders later uses of `v` after the preceding asm statement (a tcgen05.wait::ld
// that covered the load which produced `v`).
__device__ __forceinline__ void reg_fence(uint32_t (&v)[32]) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

}  // namespace idx
