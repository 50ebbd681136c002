// Host-side plumbing of libidx: status strings, the thread-local error message,
// device queries, TMA descriptor encoding, workspace sizing and the block-span
// helper. No kernels live here.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace idx {

namespace {
thread_local char g_last_error[512] = "";

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}
}  // namespace

idx_status_t fail(idx_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

idx_status_t check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    return fail(IDX_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  }
  return IDX_OK;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

int64_t device_l2_bytes() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

idx_status_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank,
                               const void* base, const uint64_t* dims,
                               const uint64_t* strides_bytes, const uint32_t* box,
                               CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(IDX_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  CUresult r = enc(map, dtype, rank, const_cast<void*>(base), gdim, gstride, bdim, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    return fail(IDX_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d, rank %d)",
                static_cast<int>(r), rank);
  }
  return IDX_OK;
}

}  // namespace idx

extern "C" {

const char* idx_status_string(idx_status_t status) {
  switch (status) {
    case IDX_OK: return "ok";
    case IDX_ERR_INVALID_ARG: return "invalid argument";
    case IDX_ERR_UNSUPPORTED: return "unsupported configuration";
    case IDX_ERR_CUDA: return "CUDA error";
    case IDX_ERR_DEVICE: return "device-side error";
  }
  return "unknown status";
}

const char* idx_last_error(void) { return idx::g_last_error; }

size_t idx_workspace_bytes(int op, int32_t rows, int32_t max_cols, int32_t k) {
  (void)k;
  switch (op) {
    case IDX_OP_MQA_LOGITS_PREFILL:
    case IDX_OP_PAGED_MQA_LOGITS_DECODE:
    case IDX_OP_TOPK:
    case IDX_OP_SPARSE_TOPK_REMAP:
      // optional first-digit histogram: 1024 uint32 counters per row; none
      // when the selection of these rows would not read it
      if (rows <= 0 || (max_cols > 0 && idx::topk_rows_short(rows, max_cols))) return 0;
      return static_cast<size_t>(rows) * 1024 * sizeof(uint32_t);
    default:
      return 0;
  }
}

idx_status_t idx_block_span(int64_t block_stride, int64_t token_stride, int32_t* span) {
  if (!span || block_stride <= 0 || token_stride <= 0) {
    return idx::fail(IDX_ERR_INVALID_ARG, "idx_block_span: strides must be positive and span non-NULL");
  }
  if (block_stride % token_stride != 0) {
    return idx::fail(IDX_ERR_UNSUPPORTED,
                     "idx_block_span: block stride %lld is not a multiple of the token stride %lld",
                     static_cast<long long>(block_stride), static_cast<long long>(token_stride));
  }
  int64_t s = block_stride / token_stride;
  if (s > INT32_MAX) return idx::fail(IDX_ERR_UNSUPPORTED, "idx_block_span: span exceeds int32");
  *span = static_cast<int32_t>(s);
  return IDX_OK;
}

idx_status_t idx_device_error(cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  long long info[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  unsigned int a = idx::logits_read_and_clear_error(stream, &e, info);
  if (e != cudaSuccess) return idx::fail(IDX_ERR_CUDA, "idx_device_error: %s", cudaGetErrorString(e));
  unsigned int b = idx::index_ops_read_and_clear_error(stream, &e);
  if (e != cudaSuccess) return idx::fail(IDX_ERR_CUDA, "idx_device_error: %s", cudaGetErrorString(e));
  unsigned int c = idx::q_rope_read_and_clear_error(stream, &e);
  if (e != cudaSuccess) return idx::fail(IDX_ERR_CUDA, "idx_device_error: %s", cudaGetErrorString(e));
  unsigned int d = idx::topk_read_and_clear_error(stream, &e);
  if (e != cudaSuccess) return idx::fail(IDX_ERR_CUDA, "idx_device_error: %s", cudaGetErrorString(e));
  unsigned int f = idx::diag_read_and_clear_error(stream, &e);
  if (e != cudaSuccess) return idx::fail(IDX_ERR_CUDA, "idx_device_error: %s", cudaGetErrorString(e));
  if (a || b || c || d || f) {
    return idx::fail(IDX_ERR_DEVICE,
                     "device error flags: logits 0x%08x (bit w: wait site w expired; first: site %lld "
                     "block %lld tile-ordinal %lld group %lld tile %lld barrier %lld parity %lld), "
                     "index ops 0x%08x (1 = a row's ks is not a multiple of sbk, 2 = a slot "
                     "beyond int32), q rope 0x%08x (1 = a position outside the cos/sin table), "
                     "top-k 0x%08x (2 = a fused slot beyond int32), diagnostics 0x%08x (1 = a wait "
                     "for the tensor core expired)",
                     a, info[0], info[1], info[2], info[3], info[4], info[5], info[6], b, c, d, f);
  }
  return IDX_OK;
}

}  // extern "C"
