/*
 * idx.h - C ABI of libidx, the GB300 (sm_103a) FP8 lightning indexer.
 *
 * The lightning indexer of DeepSeek Sparse Attention scores every query row t
 * against every visible history token s,
 *
 *     logits[t, s] = sum_{h < 64} w[t, h] * (q[t, h] . k[s])
 *
 * keeps the 2048 best tokens per row and hands their positions to the main
 * attention ("DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", section "Indexer 内部六步",
 * step 6). q is 64 heads x 128 dims of FP8 e4m3; every q-side coefficient is
 * folded into w (step 4), so the kernels multiply by no other factor. k is one
 * shared 128-dim e4m3 vector per token with one fp32 scale, stored as 132 bytes
 * per token in a paged cache (the page's cost table and data-flow item 1).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer unless stated otherwise. The
 *   caller owns every buffer; the library allocates nothing (the V4.1 review,
 *   "评论区精华": the forward pass allocates nothing, scratch is passed in).
 * - e4m3 bytes are passed as uint8_t, bf16 as uint16_t bit patterns.
 * - 2-D arguments carry an explicit row stride ("ld_*", in ELEMENTS of the
 *   argument's own type unless the name says bytes), so column slices of larger
 *   buffers work (the V4.1 review asks the kernels to take strides).
 * - Each call validates its host-side scalars and returns an idx_status_t. It
 *   never reads device memory to validate, never synchronises the stream and has
 *   no fallback path: an unsupported configuration is an error, not a slower
 *   route (the V4.1 review: fail closed, no PyTorch fallback).
 * - Work is enqueued on `stream` (0 = legacy default stream of the current
 *   device). Errors from the launch itself are reported as IDX_ERR_CUDA.
 * - Device-side problems (a bounded wait that ran out) are recorded in a device
 *   flag; idx_device_error() synchronises and reports it.
 * - idx_last_error() returns a thread-local human-readable message for the most
 *   recent non-OK status.
 *
 * Selection workspace
 * -------------------
 * The top-k's first radix pass histograms the top 10 bits of every score's
 * order-preserving key. The logits entry points can produce that histogram
 * while they write the scores, so the selection does not read the scores twice:
 * pass the same device buffer of idx_workspace_bytes(op, rows, 0, 0) bytes
 * (1024 uint32 per row, 16-byte aligned) as `ws` to a logits call and then to
 * idx_topk / idx_sparse_topk_remap (or their _slots forms) over the same rows and the same visible
 * columns (decode with next_n = 1: columns [0, ctx_len); sparse modes: [0, end)).
 * The buffer must be all zero before the logits call (clear it once after
 * allocating it); the selection zeroes every row it consumes, so the buffer is
 * ready for the next step. Supported by the kernels with one query per group:
 * dense decode with next_n = 1 and both sparse modes. ws = NULL selects the
 * two-pass selection. Rows of at most 4096 columns are selected from
 * registers in one read and never use the histogram: the selection only clears
 * a buffer it is given, and idx_workspace_bytes(op, rows, ld, k) returns 0 for
 * them, meaning pass NULL to both calls (the logits call then skips the
 * histogram and keeps more k in flight). For longer rows the histogram saves
 * the selection one sweep of each row but costs the logits call that extra k
 * in flight; on a GB300 the 128K and 32K decode steps measured faster without
 * it (281.3 against 282.3 us; 49.4 against 49.9 us).
 *
 * Paged cache layout (the "split block" layout)
 * ---------------------------------------------
 * Block b starts at byte b * block_stride_bytes of the cache. Token i of a block
 * keeps its 128 e4m3 bytes at offset i * 128 and its fp32 scale at offset
 * block_size * 128 + 4 * i. block_stride_bytes must be a multiple of 16 and at
 * least block_size * 132; rounding it up to a multiple of 512 (8704 bytes for 64
 * tokens) matches the block-stride alignment rule of the V4.1 review
 * ("实现拆解" item 4). The physical slot of a token is
 * block * block_size + offset.
 */
#ifndef IDX_H_
#define IDX_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum idx_status {
  IDX_OK = 0,
  IDX_ERR_INVALID_ARG = 1,   /* a pointer is NULL, a size is negative, a stride too small */
  IDX_ERR_UNSUPPORTED = 2,   /* well-formed but outside what the kernels implement */
  IDX_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
  IDX_ERR_DEVICE = 4         /* a kernel reported a device-side failure (idx_device_error) */
} idx_status_t;

enum { IDX_F32 = 0, IDX_BF16 = 1 };          /* element types of weights, k and logits */
enum {                                       /* k scale format, stored as fp32 in the cache */
  IDX_SCALE_FP32 = 0,                        /*   amax / 448 */
  IDX_SCALE_UE8M0 = 1                        /*   the smallest power of two >= amax / 448 */
};

/* operation codes of idx_workspace_bytes */
enum {
  IDX_OP_K_QUANT_AND_CACHE = 1,
  IDX_OP_GATHER_K = 2,
  IDX_OP_MQA_LOGITS_PREFILL = 3,
  IDX_OP_PAGED_MQA_LOGITS_DECODE = 4,
  IDX_OP_TOPK = 5,
  IDX_OP_EXPAND_CANDIDATES = 6,
  IDX_OP_SPARSE_TOPK_REMAP = 7,
  IDX_OP_REQ_TO_GLOBAL_SLOTS = 8
};

#define IDX_HEADS 64
#define IDX_HEAD_DIM 128
#define IDX_TOKEN_BYTES 132
#define IDX_MXFP4_TOKEN_BYTES 68

/*
 * idx_k_quant_and_cache - quantise k to e4m3 and insert it into the paged cache.
 *
 * "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", "Indexer 内部六步" step 5: k
 * quantisation is fused with the cache insert. Per token, in IEEE binary32:
 * amax = max_d |k_d|; scale = amax / 448; byte_d = e4m3_rn_satfinite(k_d / scale).
 * A zero scale (all-zero k, or amax / 448 underflowing) stores scale 0 and zero
 * bytes. One scale per 128 values (step 4 fixes the 128-element scale block).
 *
 *   k             [n_tok, 128] of k_dtype (IDX_BF16 or IDX_F32), row stride ld_k
 *                 elements (ld_k >= 128).
 *   slot_mapping  int64 [n_tok]: physical slot of each token; a negative slot, or
 *                 one >= num_blocks * block_size, skips the token.
 *   cache         uint8 [num_blocks, block_stride_bytes], written in place.
 *   block_size    tokens per block, one of 16, 32, 64, 128.
 *   scale_fmt     IDX_SCALE_FP32, or IDX_SCALE_UE8M0 (step 5's scale_fmt option:
 *                 the binary32 amax / 448 rounded up to a power of two, so the
 *                 division by it is exact; same 4-byte slot).
 * Errors: IDX_ERR_INVALID_ARG for NULL pointers with n_tok > 0, n_tok < 0,
 * ld_k < 128, block_stride_bytes < block_size * 132; IDX_ERR_UNSUPPORTED for
 * another block_size, block_stride_bytes % 16 != 0, another dtype or scale_fmt.
 */
idx_status_t idx_k_quant_and_cache(const void* k, int k_dtype, int64_t ld_k, int32_t n_tok,
                                   const int64_t* slot_mapping, uint8_t* cache,
                                   int32_t num_blocks, int32_t block_size,
                                   int64_t block_stride_bytes, int scale_fmt,
                                   cudaStream_t stream);

/*
 * The MXFP4 indexer cache (the V4.1 path)
 * ---------------------------------------
 * "V4.1 索引器接入稀疏 MQA logits", 功能与动机 and 实现拆解 items 1-2: the V4.1
 * consumer layers read an MXFP4 indexer cache (风险与影响: indexer_kv_dtype
 * "mxfp4") through an fp8 x fp4 MQA-logits kernel. The page prints neither the
 * format nor the layout; this library reads it as OCP MXFP4 over the 128 dims
 * of a token: four blocks of 32 dims, each element FP4 E2M1 (magnitudes 0, 0.5,
 * 1, 1.5, 2, 3, 4, 6), each block one E8M0 scale 2^(code - 127). A token takes
 * 64 element bytes plus 4 scale bytes = IDX_MXFP4_TOKEN_BYTES, about half the
 * 132 bytes of the e4m3 cache. Split block layout: block b starts at
 * b * block_stride_bytes; token i keeps its elements at i * 64 (dim d in byte
 * d / 2, even d in the low nibble) and its four scale codes at
 * block_size * 64 + 4 * i (byte j scales dims 32 j .. 32 j + 31).
 * block_stride_bytes must be at least block_size * 68 and a multiple of 32, the
 * cache 32-byte aligned; rounding the stride up to 512 (4608 bytes for 64
 * tokens) follows the V4.1 stride rule. q stays e4m3 with its scale folded into
 * the weights, so a score is
 *     sum_h w[h] * sum_d q8[h, d] * e2m1(k[d]) * 2^(E[d / 32] - 127).
 */

/*
 * idx_k_quant_and_cache_mxfp4 - quantise k to MXFP4 and insert it into an MXFP4 cache.
 *
 * "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", "Indexer 内部六步" step 5 (the
 * quantisation is fused with the insert), for the MXFP4 cache above. Per token
 * and 32-dim block, the OCP MX conversion: amax = max |k_d| in binary32; shared
 * exponent floor(log2(amax)) - 2, clamped to [-127, 127] (zero or tiny blocks get
 * -127); element = e2m1 of k_d / 2^shared, rounded to nearest even and saturated
 * to +-6 (the sign of a zero result is kept). Inputs must be finite.
 *
 *   k, ld_k, n_tok, slot_mapping, num_blocks, block_size: as idx_k_quant_and_cache.
 *   cache  uint8 [num_blocks, block_stride_bytes], written in place.
 * Errors: IDX_ERR_INVALID_ARG for NULL pointers with n_tok > 0, negative sizes,
 * ld_k < 128, block_stride_bytes < block_size * 68; IDX_ERR_UNSUPPORTED for
 * another block_size or dtype, block_stride_bytes % 32 != 0, or a cache that is
 * not 32-byte aligned.
 */
idx_status_t idx_k_quant_and_cache_mxfp4(const void* k, int k_dtype, int64_t ld_k, int32_t n_tok,
                                         const int64_t* slot_mapping, uint8_t* cache,
                                         int32_t num_blocks, int32_t block_size,
                                         int64_t block_stride_bytes, cudaStream_t stream);

enum { IDX_ROPE_NEOX = 0, IDX_ROPE_INTERLEAVED = 1 };  /* pairing of the rotary dims */

/*
 * idx_q_rope_quant - prepare the indexer's q: partial RoPE, per-head FP8
 * quantisation, and the weights with every q-side coefficient folded in.
 *
 * "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", "Indexer 内部六步" steps 3-4:
 * RoPE is applied to the first 64 of the 128 dims of each head; q is quantised
 * with one scale per 128 values (one per head); the weights absorb
 * q_scale * softmax_scale * n_head_scale, so the scoring kernels take q8 raw.
 * "V4.1 索引器接入稀疏 MQA logits", 实现拆解 item 5: the weights may be written
 * directly as bf16, the fp32 result rounded once.
 *
 * Per token t and head h, in IEEE binary32 with every operation rounded (no
 * fused multiply-add), c = cos_sin[pos, i] and s = cos_sin[pos, 32 + i] for
 * rotary pair i (pos = positions[t]):
 *   NeoX pairs (i, i + 32), interleaved pairs (2i, 2i + 1), i < 32:
 *   y_a = x_a c - x_b s,  y_b = x_b c + x_a s;   dims 64..127 pass through;
 *   scale = max_d |y_d| / 448;  q8_d = e4m3_rn_satfinite(y_d / scale) (0 if scale 0);
 *   w_out = ((w * scale) * softmax_scale) * n_head_scale.
 *
 *   q          [T, 64, 128] of q_dtype (IDX_BF16 or IDX_F32), ld_q elements
 *              between tokens (>= 8192); rows 16-byte aligned.
 *   positions  int32 [T]: a position outside [0, max_pos) writes the token as
 *              zeros and raises the device flag (idx_device_error).
 *   cos_sin    float [max_pos, ld_cs] (ld_cs >= 64): cos of the 32 pair angles,
 *              then their sin.
 *   w          [T, 64] of w_dtype, row stride ld_w >= 64.
 *   q8         uint8 [T, 64, 128], ld_q8 bytes between tokens (>= 8192, % 16 == 0).
 *   w_out      [T, 64] of w_out_dtype, row stride ld_wo >= 64.
 * Errors: IDX_ERR_INVALID_ARG for NULL pointers with T > 0, T < 0, max_pos < 1
 * or short strides; IDX_ERR_UNSUPPORTED for another dtype or rope_style, or
 * misaligned q / q8 rows.
 */
idx_status_t idx_q_rope_quant(const void* q, int q_dtype, int64_t ld_q, const int32_t* positions,
                              const float* cos_sin, int64_t ld_cs, int32_t max_pos,
                              int32_t rope_style, const void* w, int w_dtype, int64_t ld_w,
                              float softmax_scale, float n_head_scale, int32_t T, uint8_t* q8,
                              int64_t ld_q8, void* w_out, int w_out_dtype, int64_t ld_wo,
                              cudaStream_t stream);

/*
 * idx_gather_k - copy the first n_tok tokens of one request out of the cache.
 *
 * Prefill scores gathered k ("Indexer 内部六步", the prefill/decode kernel table;
 * the V4.1 review's _gather_prefill_chunk_k). Token p comes from block
 * block_table[p / block_size], offset p % block_size.
 *
 *   block_table   int32 [ceil(n_tok / block_size)] physical block ids.
 *   k8_out        uint8 [n_tok, 128] contiguous.
 *   kscale_out    float [n_tok].
 * Errors: IDX_ERR_INVALID_ARG / IDX_ERR_UNSUPPORTED as for the insert.
 */
idx_status_t idx_gather_k(const uint8_t* cache, int32_t block_size, int64_t block_stride_bytes,
                          const int32_t* block_table, int32_t n_tok,
                          uint8_t* k8_out, float* kscale_out, cudaStream_t stream);

/*
 * idx_gather_k_mxfp4 - copy the first n_tok tokens of one request out of an
 * MXFP4 cache, for the V4.1 sparse prefill (the V4.1 review, "实现拆解" item 2:
 * the builder slices the sparse buffers for every prefill chunk as well as for
 * decode, on the MXFP4 indexer cache). Token p comes from block
 * block_table[p / block_size], offset p % block_size; its 64 bytes of e2m1
 * codes and its 32-bit word of E8M0 scale codes are copied unchanged.
 *
 *   cache         as for idx_k_quant_and_cache_mxfp4 (32-byte aligned, stride a
 *                 multiple of 32).
 *   block_table   int32 [ceil(n_tok / block_size)] physical block ids.
 *   codes_out     uint8 [n_tok, 64] contiguous, 16-byte aligned (32-byte aligned
 *                 to be scored by idx_mqa_logits_prefill_mxfp4).
 *   scales_out    uint32 [n_tok], 4-byte aligned (16-byte aligned to be scored).
 * Errors: IDX_ERR_INVALID_ARG / IDX_ERR_UNSUPPORTED as for the MXFP4 insert.
 */
idx_status_t idx_gather_k_mxfp4(const uint8_t* cache, int32_t block_size, int64_t block_stride_bytes,
                                const int32_t* block_table, int32_t n_tok, uint8_t* codes_out,
                                uint32_t* scales_out, cudaStream_t stream);

/*
 * idx_mqa_logits_prefill - logits of T query rows against gathered k.
 *
 * Dense mode (sparse_idx == NULL): row t scores tokens s in [row_ks[t], row_ke[t])
 * of k8/kscale (causality is carried by the limits: a query at position p has
 * row_ke = p + 1). logits[t, s] for s in [0, S) is written: the logit inside the
 * row's range, -inf outside it.
 *
 * Sparse mode (V4.1 hierarchical variant, the V4.1 review "功能与动机" and
 * "实现拆解" item 3): sparse_idx[t, i] (i < n_si) are absolute sparse-block ids
 * in units of sbk tokens (as idx_expand_candidates produces them); column c of
 * row t scores token sparse_idx[t, c / sbk] * sbk + c % sbk when c < end[t], and
 * holds -inf otherwise. Columns [0, n_si * sbk) are written.
 *
 *   q        uint8 e4m3 [T, 64, 128]; ld_q = row stride in BYTES (multiple of 16,
 *            >= 8192); heads are contiguous 128-byte rows.
 *   w        [T, 64] of w_dtype (IDX_F32 or IDX_BF16), row stride ld_w elements.
 *   k8       uint8 [S, 128] contiguous; kscale float [S]; both 16-byte aligned.
 *   row_ks   int32 [T] or NULL (all zero); row_ke int32 [T] (dense mode).
 *   sbk      8, 16, 32, 64 or 128 (sparse mode).
 *   logits   [T, ld_out] of out_dtype (IDX_F32 or IDX_BF16).
 *   ws       NULL, or the selection workspace (see "Selection workspace" below);
 *            sparse mode only.
 * Errors: IDX_ERR_INVALID_ARG for NULL / negative / too-small strides;
 * IDX_ERR_UNSUPPORTED for misaligned q, k8 or kscale, or an sbk outside the set.
 */
idx_status_t idx_mqa_logits_prefill(const uint8_t* q, int64_t ld_q, const void* w, int w_dtype,
                                    int64_t ld_w, const uint8_t* k8, const float* kscale,
                                    int32_t S, const int32_t* row_ks, const int32_t* row_ke,
                                    int32_t T, const int32_t* sparse_idx, int64_t ld_si,
                                    int32_t n_si, const int32_t* end, int32_t sbk,
                                    void* logits, int out_dtype, int64_t ld_out,
                                    void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * idx_mqa_logits_prefill_mxfp4 - the sparse mode of idx_mqa_logits_prefill over
 * gathered MXFP4 k (idx_gather_k_mxfp4's layout), the V4.1 sparse prefill
 * ("实现拆解" items 1-2: the fp8 x fp4 sparse MQA-logits kernel on the MXFP4
 * indexer cache). Column c < end[t] of row t scores token
 * sparse_idx[t, c / sbk] * sbk + c % sbk with the block scales applied by the
 * tensor core (e4m3 q x e2m1 k); the other columns hold -inf.
 *
 *   k_codes   uint8 [S, 64] packed e2m1 codes, 32-byte aligned.
 *   k_scales  uint32 [S] words of four E8M0 codes, 16-byte aligned.
 *   sparse_idx must be given (the MXFP4 path has no dense prefill mode:
 *   IDX_ERR_UNSUPPORTED otherwise); row_ks / row_ke are not read. Every other
 *   argument, the optional workspace and the errors are those of the sparse
 *   mode of idx_mqa_logits_prefill.
 */
idx_status_t idx_mqa_logits_prefill_mxfp4(const uint8_t* q, int64_t ld_q, const void* w, int w_dtype,
                                          int64_t ld_w, const uint8_t* k_codes, const uint32_t* k_scales,
                                          int32_t S, const int32_t* row_ks, const int32_t* row_ke,
                                          int32_t T, const int32_t* sparse_idx, int64_t ld_si,
                                          int32_t n_si, const int32_t* end, int32_t sbk,
                                          void* logits, int out_dtype, int64_t ld_out,
                                          void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * idx_paged_mqa_logits_decode - decode logits read straight from the paged cache.
 *
 * "Indexer 内部六步", the prefill/decode table: decode does not gather k, it reads
 * the paged cache through the block table. Request b has next_n query rows
 * r = b * next_n + j (j < next_n); its context holds ctx_lens[b] tokens, the
 * last next_n of which are the queries themselves, so row r sees tokens
 * [0, ctx_lens[b] - next_n + j + 1).
 *
 * Dense mode (sparse_idx == NULL): logits[r, s] is written for s < ctx_lens[b]:
 * the logit where visible, -inf for the causally hidden tail; columns
 * >= ctx_lens[b] are left untouched.
 *
 * Sparse mode: as in idx_mqa_logits_prefill with k positions relative to the
 * request (row_ks = 0): column c of row r scores token
 * sparse_idx[r, c / sbk] * sbk + c % sbk of request r / next_n when c < end[r];
 * sbk must divide block_size.
 *
 *   q, w               as for prefill, rows = B * next_n.
 *   cache              uint8 [num_blocks, block_stride_bytes] (16-byte aligned).
 *   block_table        int32 [B, ld_bt]: physical block of each logical block.
 *   ctx_lens           int32 [B].
 *   next_n             1, 2 or 4 in dense mode; any value >= 1 in sparse mode.
 *   ws                 NULL, or the selection workspace (next_n = 1 or sparse mode).
 *   logits             [B * next_n, ld_out] of out_dtype; dense mode needs
 *                      ld_out >= max(ctx_lens) (not checked: ctx_lens is device data).
 *   block_table rows must cover ceil(ctx_lens[b] / block_size) blocks, and every
 *   sparse_idx entry below end must address a token inside the request.
 * Errors: as for prefill; IDX_ERR_UNSUPPORTED for another block_size or next_n.
 */
idx_status_t idx_paged_mqa_logits_decode(const uint8_t* q, int64_t ld_q, const void* w,
                                         int w_dtype, int64_t ld_w, const uint8_t* cache,
                                         int32_t num_blocks, int32_t block_size,
                                         int64_t block_stride_bytes, const int32_t* block_table,
                                         int64_t ld_bt, const int32_t* ctx_lens, int32_t B,
                                         int32_t next_n, const int32_t* sparse_idx,
                                         int64_t ld_si, int32_t n_si, const int32_t* end,
                                         int32_t sbk, void* logits, int out_dtype,
                                         int64_t ld_out, void* ws, size_t ws_bytes,
                                         cudaStream_t stream);

/*
 * idx_paged_mqa_logits_decode_mxfp4 - decode logits read from an MXFP4 cache.
 *
 * The fp8 x fp4 scoring of the V4.1 path ("V4.1 索引器接入稀疏 MQA logits",
 * 实现拆解 item 2): the same rows, modes, outputs and workspace as
 * idx_paged_mqa_logits_decode, with k read from the MXFP4 cache described
 * above (block scales applied by the tensor core, no per-token factor).
 * Dense mode supports next_n = 1; sparse mode any next_n.
 *
 *   cache   uint8 [num_blocks, block_stride_bytes] in the MXFP4 layout
 *           (32-byte aligned, stride a multiple of 32 and >= block_size * 68).
 *   other arguments as idx_paged_mqa_logits_decode.
 * Errors: as idx_paged_mqa_logits_decode; IDX_ERR_UNSUPPORTED for dense next_n
 * other than 1 or a cache layout outside the rules above.
 */
idx_status_t idx_paged_mqa_logits_decode_mxfp4(const uint8_t* q, int64_t ld_q, const void* w,
                                               int w_dtype, int64_t ld_w, const uint8_t* cache,
                                               int32_t num_blocks, int32_t block_size,
                                               int64_t block_stride_bytes,
                                               const int32_t* block_table, int64_t ld_bt,
                                               const int32_t* ctx_lens, int32_t B, int32_t next_n,
                                               const int32_t* sparse_idx, int64_t ld_si,
                                               int32_t n_si, const int32_t* end, int32_t sbk,
                                               void* logits, int out_dtype, int64_t ld_out,
                                               void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * idx_topk - per-row top-k with -1 fill.
 *
 * "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", opening section and data-flow
 * item 2: keep the k (2048) highest-scoring tokens; the index table is int32
 * and -1 marks an empty entry. Row r considers columns [row_ks[r], row_ke[r])
 * of `logits` and writes request-local indices s - row_ks[r]. When at most k
 * columns are visible all are written in column order, then -1. Otherwise the k
 * indices of the largest values are written in unspecified order; among values
 * exactly equal at the threshold an unspecified subset is kept. NaN sorts above
 * +inf.
 *
 *   logits   [rows, ld] of dtype (IDX_F32 or IDX_BF16).
 *   row_ks   int32 [rows] or NULL (all zero); row_ke int32 [rows].
 *   out      int32 [rows, ld_out], ld_out >= k.
 *   vals     NULL, or float [rows, ld_vals]: the score of each selected entry
 *            (-inf for -1 slots), e.g. the values a context-parallel rank
 *            exchanges for idx_dcp_topk_merge.
 *   ws       NULL, or the selection workspace filled by the logits call that
 *            wrote `logits` (consumed and zeroed).
 * Errors: IDX_ERR_INVALID_ARG for NULL pointers, k < 1, ld_out < k;
 * IDX_ERR_UNSUPPORTED for k > 4096.
 */
idx_status_t idx_topk(const void* logits, int dtype, int64_t ld, const int32_t* row_ks,
                      const int32_t* row_ke, int32_t rows, int32_t k, int32_t* out,
                      int64_t ld_out, float* vals, int64_t ld_vals, void* ws, size_t ws_bytes,
                      cudaStream_t stream);

/*
 * idx_dcp_topk_merge - merge per-shard top-k lists into the global top-k.
 *
 * "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解", section "几个容易踩的点": under
 * decode context parallelism each rank scores its own shard of the context and
 * the ranks exchange only their local top-k candidates, not the score matrix;
 * this is exact because a token of the global top-k is always in the local
 * top-k of the shard that holds it. Each shard of a row contributes k_local
 * (value, shard-local index) pairs (idx_topk with `vals`); candidate j of shard
 * s stands for the global position
 *     shard_offset[row * ld_off + s] + cand_idx[row, s * k_local + j] * pos_stride
 * (contiguous shards: pos_stride 1 and each shard's first position; shards that
 * deal tokens round-robin: offset = shard number, pos_stride = number of shards).
 * For every row this call takes the n_shards * k_local candidates, laid out
 * shard after shard, and writes the global positions of the k largest values,
 * in unspecified order, followed by -1 when fewer than k candidates are valid.
 *
 *   cand_vals     float [rows, ld_v]; an empty candidate (index -1) must hold -inf.
 *   cand_idx      int32 [rows, ld_i], shard-local indices, -1 = empty.
 *   shard_offset  int32 [rows, ld_off] (device); ld_off = 0 shares one vector of
 *                 n_shards offsets between all rows; NULL means every offset is 0.
 *   pos_stride    >= 1. Global positions must fit in int32.
 *   out           int32 [rows, ld_out], ld_out >= k.
 *   vals          NULL, or float [rows, ld_vals]: the merged scores (-inf for -1 slots).
 * Candidates are ranked by value alone, so a valid candidate must score above
 * -inf to be sure of beating the empty ones (in-range logits are finite).
 * Errors: IDX_ERR_INVALID_ARG for NULL pointers, too-small strides or counts
 * below 1; IDX_ERR_UNSUPPORTED for k > 4096.
 */
idx_status_t idx_dcp_topk_merge(const float* cand_vals, int64_t ld_v, const int32_t* cand_idx,
                                int64_t ld_i, const int32_t* shard_offset, int64_t ld_off,
                                int32_t n_shards, int32_t pos_stride, int32_t k_local,
                                int32_t rows, int32_t k, int32_t* out, int64_t ld_out,
                                float* vals, int64_t ld_vals, cudaStream_t stream);

/*
 * idx_expand_candidates - flatten, filter, sort, dedupe and tail-pad candidate blocks.
 *
 * The V4.1 review, "实现拆解" item 3 and the candidate-expansion snippet. Per
 * row, with R = cand_block_size / sbk and max_block = ceil((ke - ks) / sbk):
 * every candidate c >= 0 expands to the sparse blocks c * R + j (j < R); those in
 * [0, max_block) are kept, sorted ascending and deduplicated (n unique); entry
 * i < n is x_i + ks / sbk, entries i >= n repeat the last valid id (or hold
 * ks / sbk when n == 0); end = (n - 1) * sbk + min(max(ke - (x_last * sbk + ks), 1), sbk)
 * valid columns, or 0. Deduplication is this library's reading: the page sorts
 * without deduplicating and notes that duplicates only waste work in
 * production, but a duplicated block would enter the top-k twice.
 *
 *   cand          int32 [rows, ld_c] candidate block ids (n_cand used, a power of two).
 *   row_ks        int32 [rows] or NULL; every ks must be a multiple of sbk
 *                 (a row that violates this gets end = 0 and is recorded in the
 *                 device error flag).
 *   row_ke        int32 [rows].
 *   sparse_idx    int32 [rows, ld_si], n_cand * R entries written.
 *   end           int32 [rows].
 * Errors: IDX_ERR_UNSUPPORTED unless n_cand is a power of two with
 * n_cand * R <= 1024, sbk divides cand_block_size and R is a power of two.
 */
idx_status_t idx_expand_candidates(const int32_t* cand, int64_t ld_c, int32_t rows,
                                   int32_t n_cand, const int32_t* row_ks, const int32_t* row_ke,
                                   int32_t cand_block_size, int32_t sbk, int32_t* sparse_idx,
                                   int64_t ld_si, int32_t* end, cudaStream_t stream);

/*
 * idx_sparse_topk_remap - top-k over sparse columns, then map columns to positions.
 *
 * The V4.1 review, "实现拆解" item 3 (top-k on the sparse logits, then the remap
 * kernel maps each sparse column back to its request-local position) and the
 * rows-metadata snippet (col_indices holds the column top-k). Row r selects
 * among columns [0, end[r]) exactly as idx_topk does, writes the chosen columns
 * to col_scratch (if not NULL) and the positions
 * (sparse_idx[r, c / sbk] - row_ks[r] / sbk) * sbk + c % sbk to `positions`;
 * empty entries are -1 in both.
 *
 *   sparse_logits  [rows, ld] of dtype (IDX_BF16 as the V4.1 path uses, or IDX_F32).
 *   row_ks         int32 [rows] or NULL.
 * Errors: as for idx_topk.
 */
idx_status_t idx_sparse_topk_remap(const void* sparse_logits, int dtype, int64_t ld,
                                   const int32_t* end, const int32_t* sparse_idx, int64_t ld_si,
                                   const int32_t* row_ks, int32_t sbk, int32_t rows, int32_t k,
                                   int32_t* col_scratch, int64_t ld_col, int32_t* positions,
                                   int64_t ld_pos, void* ws, size_t ws_bytes,
                                   cudaStream_t stream);

/*
 * idx_req_to_global_slots - request-local positions to physical cache slots.
 *
 * "DeepSeek V3.2 ...", section "几个容易踩的点": the indexer emits positions
 * inside the request, the attention kernel needs paged-cache slots. The DSV4
 * packed-KV fix ("修复 DSV4 FlashInfer 稀疏 MLA 在打包 KV 布局下的地址错误",
 * 实现拆解 and the remap snippet) generalises the slot to
 * block * block_span + offset for pools whose blocks hold block_span >= block_size
 * token strides. Entry v >= 0 of row r becomes
 * block_table[req(r), v / block_size] * block_span + v % block_size; negative
 * entries, and entries whose block index v / block_size >= ld_bt, become -1.
 *
 *   local        int32 [rows, ld_l], k entries per row.
 *   row_to_req   int32 [rows] or NULL (row r belongs to request r).
 *   block_table  int32 [*, ld_bt].
 *   slots        int32 [rows, ld_s]. May alias `local` when ld_s == ld_l.
 * Errors: IDX_ERR_UNSUPPORTED when block_span < block_size.
 */
idx_status_t idx_req_to_global_slots(const int32_t* local, int64_t ld_l, int32_t rows, int32_t k,
                                     const int32_t* row_to_req, const int32_t* block_table,
                                     int64_t ld_bt, int32_t block_size, int32_t block_span,
                                     int32_t* slots, int64_t ld_s, cudaStream_t stream);

/*
 * idx_topk_slots / idx_sparse_topk_remap_slots - the selection with the slot
 * conversion fused into its output pass.
 *
 * Same selection and outputs as idx_topk (without `vals`) and
 * idx_sparse_topk_remap, and in addition every request-local entry v of row r
 * converted exactly as idx_req_to_global_slots does with the same row_to_req,
 * block_table, ld_bt, block_size and block_span, written to slots[r, i]
 * (int32 [rows, ld_slots], ld_slots >= k; -1 where the entry is -1). One launch
 * instead of two; the results equal the two-call sequence. A slot beyond int32
 * is written as -1 and raises the device flag (idx_device_error).
 * Errors: those of the two calls it replaces.
 */
idx_status_t idx_topk_slots(const void* logits, int dtype, int64_t ld, const int32_t* row_ks,
                            const int32_t* row_ke, int32_t rows, int32_t k, int32_t* out,
                            int64_t ld_out, const int32_t* row_to_req, const int32_t* block_table,
                            int64_t ld_bt, int32_t block_size, int32_t block_span, int32_t* slots,
                            int64_t ld_slots, void* ws, size_t ws_bytes, cudaStream_t stream);

idx_status_t idx_sparse_topk_remap_slots(const void* sparse_logits, int dtype, int64_t ld,
                                         const int32_t* end, const int32_t* sparse_idx,
                                         int64_t ld_si, const int32_t* row_ks, int32_t sbk,
                                         int32_t rows, int32_t k, int32_t* col_scratch,
                                         int64_t ld_col, int32_t* positions, int64_t ld_pos,
                                         const int32_t* row_to_req, const int32_t* block_table,
                                         int64_t ld_bt, int32_t block_size, int32_t block_span,
                                         int32_t* slots, int64_t ld_slots, void* ws,
                                         size_t ws_bytes, cudaStream_t stream);

/*
 * idx_paged_mqa_topk_decode_noalloc - decode scoring and top-k for callers that
 * cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point; it exists for callers of
 * this library that are not allowed to call cudaMalloc: code that runs inside
 * an engine which plans every device buffer ahead of time and forbids new
 * allocations while it serves, or a plugin that is handed raw device pointers
 * and no allocator. Such callers cannot provide the selection workspace, so
 * this call keeps it in a scratch array built into the library (4 KB per row,
 * IDX_NOALLOC_MAX_ROWS rows = 4 MB on every device that loads the library,
 * held until the process exits). It allocates nothing and frees nothing.
 *
 * It computes exactly what idx_paged_mqa_logits_decode (dense mode, next_n = 1,
 * fp32 logits) followed by idx_topk over columns [0, ctx_lens[b]) compute,
 * writing the scores to `logits` [B, ld_logits] and the top-k request-local
 * indices (-1 filled) to `out` [B, ld_out]; the other arguments are as for
 * idx_paged_mqa_logits_decode.
 *
 * Every call asks the runtime for the scratch array's device address on the
 * current device (a host-side query, no allocation; asked anew each time, so
 * a context destroyed and re-created, e.g. by cudaDeviceReset, is followed
 * correctly). The first call on a device is also where the runtime sets the
 * array up there: make that first call before any stream capture. Every call
 * clears the scratch rows it uses before scoring. All calls on a device share
 * the one array, so calls whose work overlaps on the GPU (other streams, other
 * host threads) race on it and must be serialised by the caller.
 * Errors: IDX_ERR_UNSUPPORTED when B > IDX_NOALLOC_MAX_ROWS or k > 4096;
 * IDX_ERR_INVALID_ARG for k < 1, ld_out < k or NULL out / logits, all checked
 * before any work is enqueued; otherwise those of the two entry points it runs.
 */
#define IDX_NOALLOC_MAX_ROWS 1024
idx_status_t idx_paged_mqa_topk_decode_noalloc(const uint8_t* q, int64_t ld_q, const void* w,
                                               int w_dtype, int64_t ld_w, const uint8_t* cache,
                                               int32_t num_blocks, int32_t block_size,
                                               int64_t block_stride_bytes,
                                               const int32_t* block_table, int64_t ld_bt,
                                               const int32_t* ctx_lens, int32_t B, float* logits,
                                               int64_t ld_logits, int32_t k, int32_t* out,
                                               int64_t ld_out, cudaStream_t stream);

/*
 * idx_block_span - tokens per physical block of a pool (host only).
 *
 * The DSV4 packed-KV fix, 实现拆解 item 1: block_span = block_stride /
 * token_stride, rejected when it does not divide exactly.
 * Returns IDX_ERR_UNSUPPORTED (span untouched) when it does not divide,
 * IDX_ERR_INVALID_ARG for non-positive strides or a NULL span.
 */
idx_status_t idx_block_span(int64_t block_stride, int64_t token_stride, int32_t* span);

/*
 * idx_diag_mma_peak - diagnostic: keep every SM's tensor core busy with dense MMAs.
 *
 * Not part of the indexer's path: a measurement aid for the roofline of the
 * tensor-bound prefill scoring, whose denominator is this GPU's dense FP8
 * tensor-core rate. Launches `ctas` persistent CTAs (<= 0: one per SM), each
 * issuing `iters` back-to-back tcgen05.mma of shape 128 x 256 x K from fixed
 * shared-memory operands into tensor memory (kind IDX_DIAG_E4M3: e4m3 x e4m3,
 * K = 32; IDX_DIAG_BF16: bf16 x bf16, K = 16; fp32 accumulation). The caller
 * times the launch on `stream`; *flop_out (if not NULL) receives the FLOP it
 * performs, 2 * 128 * 256 * K * iters * ctas. Allocates nothing; every wait is
 * bounded (idx_device_error reports an expired one).
 * Errors: IDX_ERR_UNSUPPORTED for another kind; IDX_ERR_INVALID_ARG for
 * iters < 1 or more CTAs than SMs.
 */
enum { IDX_DIAG_E4M3 = 0, IDX_DIAG_BF16 = 1 };
idx_status_t idx_diag_mma_peak(int kind, int32_t iters, int32_t ctas, double* flop_out, cudaStream_t stream);

/*
 * idx_diag_l2_read - diagnostic: read a device buffer with every SM.
 *
 * Not part of the indexer's path: the denominator for kernels that stream data
 * L2 already holds (the sparse prefill reads its gathered k from L2 once per
 * query row; the selection reads scores the scoring kernel just wrote).
 * Launches `ctas` CTAs of 1024 threads (<= 0: one per SM). The buffer is cut
 * into `ctas` contiguous chunks; in each of `passes` passes every CTA reads one
 * chunk, a different one in consecutive passes (CTA b in pass k reads chunk
 * (b + 77 k) mod ctas), with 16-byte loads that bypass L1, four in flight per
 * thread. The caller times the launch on
 * `stream`: for a buffer that fits in L2 and was read once before, that is the
 * L2 read rate, bytes * passes / time. Allocates nothing and writes nothing the
 * caller can see. `buf` 16-byte aligned device memory of at least `bytes`.
 * Errors: IDX_ERR_INVALID_ARG for a NULL or unaligned buffer, bytes not a
 * positive multiple of 16, passes < 1, or more CTAs than SMs.
 */
idx_status_t idx_diag_l2_read(const void* buf, int64_t bytes, int32_t passes, int32_t ctas,
                              cudaStream_t stream);

/*
 * Bytes of the optional selection workspace of an operation for `rows` rows
 * (host only). max_cols = 0: the size of the buffer, whatever the row length;
 * max_cols > 0 (the `ld` the selection will be given): 0 when the selection of
 * such rows would not read the histogram on the current device (see "Selection
 * workspace"), so no buffer is needed.
 */
size_t idx_workspace_bytes(int op, int32_t rows, int32_t max_cols, int32_t k);

/* Static description of a status code (host only). */
const char* idx_status_string(idx_status_t status);

/* Thread-local message of the most recent non-OK status on this thread (host only). */
const char* idx_last_error(void);

/*
 * idx_device_error - synchronise `stream`, then read and clear the device-side
 * error flag of the current device. Returns IDX_OK when no kernel recorded a
 * failure, IDX_ERR_DEVICE (message in idx_last_error) when one did, and
 * IDX_ERR_CUDA when the synchronisation itself failed.
 */
idx_status_t idx_device_error(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H_ */
