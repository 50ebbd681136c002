// Allocation-free decode scoring + selection.
//
// The fused selection needs a per-row histogram workspace between the logits
// kernel and the top-k kernel. Callers that cannot allocate device memory
// cannot provide one, so this file keeps that workspace in a fixed array that
// is part of the library image: it exists on every device that loads the
// library, for as long as the library stays loaded, and it is never allocated
// or freed by a call.
#include "common.cuh"

namespace idx {
namespace {

constexpr int kNoAllocMaxRows = IDX_NOALLOC_MAX_ROWS;
constexpr int kHistWordsPerRow = 1024;  // first-digit bins of the selection

// Shared by every call on a device. The selection re-zeroes each row it
// consumes, and every call clears the rows it uses before scoring, so stale
// contents from an earlier (possibly failed) call are never read.
static __device__ __align__(256) uint32_t g_noalloc_hist[kNoAllocMaxRows * kHistWordsPerRow];

// Device address of the scratch array on the current device. In host code the
// array's name only stands in for the symbol; the address the kernels need is
// asked of the runtime with the device current. It is asked on every call, not
// cached: a context torn down and created again (cudaDeviceReset) places the
// array at a new address, and the query is a host-side lookup that allocates
// nothing.
idx_status_t scratch_for_current_device(const char* fn, uint32_t** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_hist);
  if (e != cudaSuccess || !ptr) {
    return fail(IDX_ERR_CUDA, "%s: cudaGetSymbolAddress of the scratch array: %s", fn,
                cudaGetErrorString(e));
  }
  *out = static_cast<uint32_t*>(ptr);
  return IDX_OK;
}

}  // namespace
}  // namespace idx

using namespace idx;

extern "C" idx_status_t idx_paged_mqa_topk_decode_noalloc(
    const uint8_t* q, int64_t ld_q, const void* w, int w_dtype, int64_t ld_w, const uint8_t* cache,
    int32_t num_blocks, int32_t block_size, int64_t block_stride_bytes, const int32_t* block_table,
    int64_t ld_bt, const int32_t* ctx_lens, int32_t B, float* logits, int64_t ld_logits, int32_t k,
    int32_t* out, int64_t ld_out, cudaStream_t stream) {
  const char* fn = "idx_paged_mqa_topk_decode_noalloc";
  if (B < 0) return fail(IDX_ERR_INVALID_ARG, "%s: B < 0", fn);
  if (B > kNoAllocMaxRows) {
    return fail(IDX_ERR_UNSUPPORTED,
                "%s: %d rows exceed the %d rows its built-in scratch array holds; use "
                "idx_paged_mqa_logits_decode + idx_topk with a caller workspace instead",
                fn, B, kNoAllocMaxRows);
  }
  // the selection's own checks, made before any work is enqueued so that a bad
  // k or output never leaves a call half done (scores written, no selection)
  if (k < 1 || k > 4096) {
    return fail(k < 1 ? IDX_ERR_INVALID_ARG : IDX_ERR_UNSUPPORTED, "%s: k %d outside [1, 4096]", fn, k);
  }
  if (ld_out < k) return fail(IDX_ERR_INVALID_ARG, "%s: ld_out < k", fn);
  if (B == 0) return IDX_OK;
  if (!out || !logits) return fail(IDX_ERR_INVALID_ARG, "%s: NULL out or logits", fn);
  uint32_t* hist = nullptr;
  idx_status_t st = scratch_for_current_device(fn, &hist);
  if (st != IDX_OK) return st;
  const size_t bytes = static_cast<size_t>(B) * kHistWordsPerRow * sizeof(uint32_t);
  // the histogram rows must start at zero; cudaMemsetAsync writes, it does not allocate
  cudaError_t e = cudaMemsetAsync(hist, 0, bytes, stream);
  if (e != cudaSuccess) return fail(IDX_ERR_CUDA, "%s: clearing the scratch: %s", fn, cudaGetErrorString(e));
  st = idx_paged_mqa_logits_decode(q, ld_q, w, w_dtype, ld_w, cache, num_blocks, block_size,
                                   block_stride_bytes, block_table, ld_bt, ctx_lens, B, 1, nullptr,
                                   0, 0, nullptr, 0, logits, IDX_F32, ld_logits, hist, bytes, stream);
  if (st != IDX_OK) return st;
  return idx_topk(logits, IDX_F32, ld_logits, nullptr, ctx_lens, B, k, out, ld_out, nullptr, 0, hist,
                  bytes, stream);
}
