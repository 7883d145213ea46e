/*
 * sparse_mla.h -- C ABI of the GB300 (sm_103a) DSA sparse-MLA attention forward.
 *
 * The operation (all three entry points).  For every query token t and
 * query head h, over the token's list of top-k KV indices:
 *
 *   valid entries  j : index != -1 and inside the token's KV range
 *   s_j      = sm_scale * sum_{d<576} q[t,h,d] * kv[row_j, d]
 *   lse[t,h] = ln sum_j exp(s_j)                  (natural log, fp32)
 *   out[t,h] = sum_j exp(s_j - lse[t,h]) * kv[row_j, 0:512]   (bf16)
 *
 * One latent KV head of 576 bf16 values per token is shared by every query
 * head; its first 512 values are the value ("[Feature] Add optional FlashMLA
 * backend for DSA Sparse MLA", Runtime constraints: kv_group=1,
 * value_dim=512).  The shapes d_qk=576, d_v=512, topk=2048 at 8 TP-local
 * heads are the isolated-forward workload of "feat: add XTuner TileLang
 * sparse MLA backend" (Performance), whose Validation section covers
 * -1-padded index lists; the same page's Summary has one kernel serve
 * packed prefill and zero-copy BF16 paged-cache decode.  Output and LSE are
 * the two results the FlashMLA page aligns across implementations
 * (Motivation).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never frees or retains them.  Tensors are dense row-major.
 *   - q, kv / kv_cache and out must be 16-byte aligned; index, length and
 *     lse arrays 4-byte aligned.
 *   - Entries are taken with multiplicity (a repeated index counts once per
 *     occurrence).  Index VALUES are never an error: -1, any other negative
 *     value and anything at or past the token's KV length is masked and the
 *     masked row is never read.  A token with no valid entry gets out = 0
 *     and lse = -inf.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream): no host synchronisation, no allocation.  The first
 *     call on a device performs one-time set-up (device query, kernel
 *     attributes) and should not be made during stream capture.
 *   - Errors: arguments are checked on the host before any launch and a
 *     non-OK status means nothing was launched, except SPARSE_MLA_ERR_CUDA
 *     after a failed launch.  No exception or abort crosses the ABI.
 *   - Supported device: compute capability 10.3 (GB300); other devices get
 *     SPARSE_MLA_ERR_UNSUPPORTED_ARCH.  d_qk must be 576 and d_v 512
 *     (SPARSE_MLA_ERR_UNSUPPORTED_SHAPE otherwise).  Any h_q >= 1 and
 *     topk >= 1 are accepted.
 *   - Device-side waits are bounded.  A kernel whose wait expires records a
 *     code in a per-device error word (sparse_mla_get_device_error), leaves
 *     its outputs undefined and returns; later launches on that device do no
 *     work until the word is cleared.
 */
#ifndef SPARSE_MLA_H
#define SPARSE_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPARSE_MLA_OK = 0,
  SPARSE_MLA_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, negative size, bad count */
  SPARSE_MLA_ERR_UNSUPPORTED_SHAPE = 2,  /* d_qk != 576 or d_v != 512 */
  SPARSE_MLA_ERR_UNSUPPORTED_ARCH = 3,   /* current device is not sm_103 */
  SPARSE_MLA_ERR_CUDA = 4,               /* a CUDA runtime/driver call or launch failed */
  SPARSE_MLA_ERR_DEVICE_TIMEOUT = 5,     /* reported by sparse_mla_get_device_error */
  SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL = 6 /* decode workspace below sparse_mla_decode_workspace_size */
} sparse_mla_status_t;

/*
 * Dense-layout forward (prefill over one sequence or any token batch).
 *
 *   q        bf16 [s_q, h_q, d_qk]
 *   kv       bf16 [s_kv, d_qk]      (the [s_kv, 1, d_qk] single-head layout)
 *   indices  int32 [s_q, topk]      (the [s_q, 1, topk] layout); row index
 *                                   into kv, -1 padded; valid iff 0 <= i < s_kv
 *   sm_scale score scale (1/sqrt(576) for the pages' workloads)
 *   out      bf16 [s_q, h_q, d_v]   written
 *   lse      fp32 [s_q, h_q]        written, natural log
 *
 * s_q == 0 is a no-op.  s_kv == 0 masks everything.
 */
sparse_mla_status_t sparse_mla_fwd(const void* q, const void* kv, const int32_t* indices, float sm_scale,
                                   void* out, float* lse, int s_q, int s_kv, int h_q, int d_qk, int d_v,
                                   int topk, void* stream);

/*
 * Backward of sparse_mla_fwd_varlen (packed sequences; indices local to each
 * token's sequence, as there).  Arguments as for sparse_mla_bwd, with the
 * packed layout of sparse_mla_fwd_varlen: dq fp32 [total_q, h_q, d_qk]
 * written, dkv fp32 [total_kv, d_qk] zeroed then accumulated.
 */
sparse_mla_status_t sparse_mla_bwd_varlen(const void* q, const void* kv, const int32_t* indices,
                                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                                          const void* out, const float* lse, const void* dout, float sm_scale,
                                          float* dq, float* dkv, int total_q, int total_kv, int h_q, int d_qk,
                                          int d_v, int topk, void* stream);

/*
 * Indices-free causal forward for short prefill, where the top-k selection
 * keeps every causal position ("feat: add XTuner TileLang sparse MLA
 * backend", Summary: short prefill), so no index tensor is needed.  The s_q
 * queries are the last s_q of the s_kv positions: query t attends to every
 * kv row at or before position t + s_kv - s_q (a query before position 0
 * attends to nothing: out = 0, LSE = -inf).  The result equals
 * sparse_mla_fwd given those positions as each token's list.
 *
 *   q        bf16 [s_q, h_q, d_qk]
 *   kv       bf16 [s_kv, d_qk]
 *   out      bf16 [s_q, h_q, d_v]   written
 *   lse      fp32 [s_q, h_q]        written, natural log
 *
 * s_q == 0 is a no-op.  s_kv == 0 masks everything.
 */
sparse_mla_status_t sparse_mla_fwd_causal(const void* q, const void* kv, float sm_scale, void* out, float* lse,
                                          int s_q, int s_kv, int h_q, int d_qk, int d_v, void* stream);

/*
 * Backward of sparse_mla_fwd: gradients with respect to q and kv for an
 * upstream gradient dout of out (the LSE output carries no gradient), the
 * pass the training users pair with the forward (prime-rl cudnn_flashmla
 * page: sparse-attention forward and backward timings).  Per token, with P
 * the attention weights over its valid rows K (V = K[:, :512]):
 *   dS = P * (dout V^T - rowsum(dout * out)),  dq = sm_scale dS K,
 *   dkv[row] += sm_scale dS^T q  (all 576 columns)  +  P^T dout (first 512).
 *
 *   q, kv, indices, sm_scale   as for sparse_mla_fwd
 *   out      bf16 [s_q, h_q, d_v]   the forward's output
 *   lse      fp32 [s_q, h_q]        the forward's LSE
 *   dout     bf16 [s_q, h_q, d_v]
 *   dq       fp32 [s_q, h_q, d_qk]  written
 *   dkv      fp32 [s_kv, d_qk]      written (zeroed on the stream, then accumulated)
 *
 * Rows listed by several tokens accumulate every contribution (atomic adds:
 * the summation order, hence the last bits of dkv, varies between calls).
 */
sparse_mla_status_t sparse_mla_bwd(const void* q, const void* kv, const int32_t* indices, const void* out,
                                   const float* lse, const void* dout, float sm_scale, float* dq, float* dkv,
                                   int s_q, int s_kv, int h_q, int d_qk, int d_v, int topk, void* stream);

/*
 * Packed (varlen) prefill: `batch` sequences concatenated along the token
 * axis.  Token t belongs to the sequence b with cu_seqlens_q[b] <= t <
 * cu_seqlens_q[b+1]; its indices are LOCAL to that sequence: entry i reads
 * kv row cu_seqlens_kv[b] + i and is valid iff
 * 0 <= i < cu_seqlens_kv[b+1] - cu_seqlens_kv[b].
 *
 *   q             bf16 [total_q, h_q, d_qk]
 *   kv            bf16 [total_kv, d_qk]
 *   indices       int32 [total_q, topk]
 *   cu_seqlens_q  int32 [batch+1] device, non-decreasing, cu_seqlens_q[0] = 0,
 *                 cu_seqlens_q[batch] = total_q
 *   cu_seqlens_kv int32 [batch+1] device, same rules against total_kv
 *   out / lse     as sparse_mla_fwd with s_q = total_q
 *
 * Rows computed from malformed cu_seqlens_kv that fall outside [0, total_kv)
 * are masked, never read.
 */
sparse_mla_status_t sparse_mla_fwd_varlen(const void* q, const void* kv, const int32_t* indices,
                                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                                          int batch, float sm_scale, void* out, float* lse, int total_q,
                                          int total_kv, int h_q, int d_qk, int d_v, int topk,
                                          void* stream);

/*
 * Bytes of device workspace sparse_mla_decode needs for this shape on the
 * current device (0 when it needs none).  The value depends on the device's
 * SM count; query it on the device that will run the call.
 */
size_t sparse_mla_decode_workspace_size(int batch, int s_next, int h_q, int d_v, int topk);

/*
 * Decode over a paged BF16 KV cache, read in place.
 *
 *   q             bf16 [batch, s_next, h_q, d_qk]   s_next query tokens per request
 *                 (the speculative tokens of a request, e.g. 6 for MTP5)
 *   kv_cache      bf16 [num_blocks, page_size, d_qk]
 *   block_table   int32 [batch, max_blocks]: page of logical block k of request b
 *   cache_seqlens int32 [batch]: tokens in request b's cache
 *   indices       int32 [batch, s_next, topk]: LOGICAL positions in the request;
 *                 entry i is valid iff 0 <= i < cache_seqlens[b], i / page_size <
 *                 max_blocks and the page entry lies in [0, num_blocks); it reads
 *                 cache slot block_table[b][i / page_size] * page_size + i % page_size
 *   out           bf16 [batch, s_next, h_q, d_v]
 *   lse           fp32 [batch, s_next, h_q]
 *   workspace     device buffer of at least sparse_mla_decode_workspace_size(...)
 *                 bytes, 16-byte aligned (may be NULL when that size is 0);
 *                 contents ignored on entry.  The library writes per-split
 *                 partial results and one arrival counter per (token, 64-head
 *                 group, softmax group) there during the call (the counters
 *                 are zeroed on the call's stream before the kernel).  Two
 *                 calls that may run concurrently need separate workspaces.
 *
 * num_blocks * page_size must fit in int32.
 */
sparse_mla_status_t sparse_mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                                      const int32_t* cache_seqlens, const int32_t* indices, float sm_scale,
                                      void* out, float* lse, int batch, int s_next, int h_q, int d_qk,
                                      int d_v, int topk, int page_size, int max_blocks, int num_blocks,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * sparse_mla_decode over an FP8 paged KV cache, read in place.  The pages
 * name this path ("feat: add XTuner TileLang sparse MLA backend", Summary:
 * the FP8 MLA KV-cache path; Pull request overview: BF16 and FP8 sparse
 * decode tests for FlashMLA) without its format; the format is the FP8
 * sparse-decode cache published with DeepSeek-V3.2's FlashMLA kernels.  One
 * cache slot (one token's latent row) is 656 bytes:
 *
 *   bytes [0, 512)    512 float8 e4m3 codes (OCP E4M3, the variant without
 *                     infinities) of the latent's first 512 values;
 *   bytes [512, 528)  4 fp32 scales; scale k applies to codes 128k .. 128k+127;
 *   bytes [528, 656)  the latent's last 64 values (rope), bf16.
 *
 * The row the attention uses is code * scale (d < 512) and the rope values.
 * Arithmetic:
 *   h_q <= 16   the tensor cores contract the codes themselves, as bf16
 *               values code * 2^-120 (exact; e4m3 subnormals become bf16
 *               subnormals): each 128-column tile's partial score is taken
 *               back by the row's tile scale (and 2^120) in fp32, and P.V
 *               takes, per tile, P times the row's tile scale and 2^88
 *               rounded to bf16 (its sum scaled back by 2^32).  Tile scales
 *               below 2^32 keep these finite.  A NaN code (0x7F, 0xFF) under
 *               a finite scale is read as +-480; a NaN scale gives NaN.
 *   h_q > 16    each gathered row is dequantized to bf16 (code * scale in
 *               fp32, round to nearest even) in shared memory, then computed
 *               as sparse_mla_decode does.
 *
 *   kv_cache      uint8 [num_blocks, page_size, 656], 16-byte aligned
 *   everything else, including the workspace (sparse_mla_decode_workspace_size),
 *   as sparse_mla_decode.
 */
sparse_mla_status_t sparse_mla_decode_fp8(const void* q, const void* kv_cache, const int32_t* block_table,
                                          const int32_t* cache_seqlens, const int32_t* indices, float sm_scale,
                                          void* out, float* lse, int batch, int s_next, int h_q, int d_qk, int d_v,
                                          int topk, int page_size, int max_blocks, int num_blocks, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * sparse_mla_decode without a caller workspace, for callers that cannot
 * allocate device memory at the point of the call: code running inside a
 * serving engine whose allocator owns every byte of the device (a KV-cache
 * pool sized to fill HBM, with allocation forbidden after start-up), plug-ins
 * that receive device pointers from a host runtime but have no allocator of
 * their own, and hot paths that must not call cudaMalloc because it can
 * synchronise the device.  The pages describe no counterpart of this entry
 * point; it exists for such callers only.
 *
 * Arguments, layouts and results are those of sparse_mla_decode, minus the
 * workspace.  The per-split partial results go to one scratch array of
 * sparse_mla_decode_noalloc_max_scratch_bytes() bytes (8 MiB) that the
 * library holds in device memory on every GPU that loads it, until the
 * process exits.  The arguments are checked first, exactly as
 * sparse_mla_decode checks them (same status codes); then a shape whose
 * sparse_mla_decode_workspace_size exceeds that maximum is rejected with
 * SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL before any launch (use
 * sparse_mla_decode with a workspace for it).  The partials take
 * 2 x CTAs x min(h_q, 64) x 513 x 4 bytes, rounded up to 16, and the merge
 * counters 8 bytes per (token, 64-head group): on a 152-SM GB300 with a full
 * grid (any batch x s_next >= 10 at topk 2048) h_q <= 13 fits for up to
 * 34,000 tokens, so the 8-head MTP decode does, while h_q >= 14 fits only
 * for grids small enough (few tokens, short lists).  The call makes no cudaMalloc, cudaFree or
 * other allocating call.
 *
 * Every call shares the one scratch array, which keeps the last call's
 * contents; each call overwrites every entry it later reads, so nothing has
 * to be cleared.  Calls whose kernels overlap on the GPU (different streams,
 * or different host threads) race on the array: serialise them.  The first
 * call on a device looks up the array's device address once (with that device
 * current); make that first call before any stream capture.
 */
sparse_mla_status_t sparse_mla_decode_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                                              const int32_t* cache_seqlens, const int32_t* indices, float sm_scale,
                                              void* out, float* lse, int batch, int s_next, int h_q, int d_qk,
                                              int d_v, int topk, int page_size, int max_blocks, int num_blocks,
                                              void* stream);

/* Size in bytes of the scratch array sparse_mla_decode_noalloc uses. */
size_t sparse_mla_decode_noalloc_max_scratch_bytes(void);

/*
 * Debug exports of "which entries are masked": counts[t] (int32, written) is
 * the number of valid entries of token t's list, with multiplicity, as the
 * forward gathers them.  Each call runs the forward's own gather walk (its
 * item schedule, 64-entry block scan and skip, index -> row mapping and
 * validity test) with the copies and the arithmetic left out, so the count is
 * that of the rows the forward reads, to be compared exactly with the
 * definition's count of valid entries ("feat: add XTuner TileLang sparse
 * MLA backend", Validation: -1-padded index lists).  Arguments are
 * those of the matching forward (sparse_mla_fwd, sparse_mla_fwd_varlen,
 * sparse_mla_decode); counts int32 [tokens], 4-byte aligned, device.  Nothing
 * is allocated; launches on `stream`.
 */
sparse_mla_status_t sparse_mla_debug_valid_count(const int32_t* indices, int s_q, int s_kv, int topk,
                                                 int32_t* counts, void* stream);
sparse_mla_status_t sparse_mla_debug_valid_count_varlen(const int32_t* indices, const int32_t* cu_seqlens_q,
                                                        const int32_t* cu_seqlens_kv, int batch, int total_q,
                                                        int total_kv, int topk, int32_t* counts, void* stream);
sparse_mla_status_t sparse_mla_debug_valid_count_paged(const int32_t* indices, const int32_t* block_table,
                                                       const int32_t* cache_seqlens, int batch, int s_next, int topk,
                                                       int page_size, int max_blocks, int num_blocks,
                                                       int32_t* counts, void* stream);

/* ------------------------------------------------------------------------
 * DSA indexer: the step that produces the index lists above.
 *
 * The pages name the indexer and its top-k ("[Feature] Add optional FlashMLA
 * backend for DSA Sparse MLA", Changes: the TileLang indexer; "feat: add
 * XTuner TileLang sparse MLA backend", Summary: DSA index production for
 * short prefill, Copilot overview: prefill scores in query-row chunks under a
 * logits budget) without printing its formula.  It is read as the DSA
 * lightning indexer published with DeepSeek-V3.2: for query row t with
 * indexer heads j < h_idx and one key per KV position s,
 *
 *   I[t,s] = sum_j weights[t,j] * max(0, q_idx[t,j,:] . k_idx[s,:])
 *
 * computed from bf16 q_idx and k_idx with fp32 accumulation and fp32
 * weights.  Visibility is causal with the queries of a sequence at its end:
 * local row t of a sequence with lq query rows and lk KV positions sees
 * positions 0 .. t + lk - lq, i.e. V(t) = clip(t + lk - lq + 1, 0, lk).  Its
 * list holds the topk visible positions of largest score, equal scores
 * ranked by position (smaller first), in increasing position order, padded
 * with -1; a row with V(t) <= topk lists 0 .. V(t)-1 and is never scored.
 * A position scoring -inf is never selected (a row with fewer than topk
 * other positions lists those and pads with -1).
 * Positions are local to the row's sequence, the convention of
 * sparse_mla_fwd_varlen.
 *
 * Layout (all device pointers, row-major):
 *   q_idx    bf16 [total_q, h_idx, d_idx]       16-byte aligned
 *   k_idx    bf16 [total_kv, d_idx]             16-byte aligned
 *   weights  fp32 [total_q, h_idx]              16-byte aligned
 *   cu_seqlens_q / cu_seqlens_kv  int32 [batch + 1] packed-sequence offsets,
 *            or both NULL for one dense sequence (total_q queries at the end
 *            of total_kv positions; batch is then ignored).
 * h_idx must be 16, 32 or 64 and d_idx 128 (else
 * SPARSE_MLA_ERR_UNSUPPORTED_SHAPE); batch may not exceed 2048.  Offsets
 * are trusted; a sequence longer than the caller's row length is cut to it
 * and the device error word records 0x611.
 * ------------------------------------------------------------------------ */

/*
 * Indexer scores of query rows row0 .. row0 + n_rows - 1 (the product path of
 * dsa_indexer_topk, exported for testing and for callers that keep the
 * logits).  Row r's scores for its positions 0 .. V-1 go to
 * scores[(r - row0) * row_stride + s] (fp32); entries past V, and every
 * entry of a row with V <= skip_len, are left as they were.  row_stride must
 * be at least the longest visible length (else see above).  Nothing is
 * allocated; launches on `stream`.
 */
sparse_mla_status_t dsa_indexer_scores(const void* q_idx, const void* k_idx, const float* weights,
                                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                                       int total_q, int total_kv, int h_idx, int d_idx, int row0, int n_rows,
                                       int skip_len, float* scores, long long row_stride, void* stream);

/*
 * Selection alone: the lists of rows row0 .. row0 + n_rows - 1 from their
 * scores (layout of dsa_indexer_scores), written to
 * indices[r * topk .. r * topk + topk - 1] (int32).  Rows with V <= topk get
 * the identity list and their scores are not read (scores may be NULL when
 * no row is longer).  Scores are compared as fp32; a NaN with the sign bit
 * clear ranks above +inf.  A score of -inf (or a NaN with the sign bit set)
 * is never selected: a row with fewer selectable positions than topk lists
 * them all and pads with -1.
 */
sparse_mla_status_t dsa_topk(const float* scores, long long row_stride, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_kv, int batch, int total_q, int total_kv, int row0,
                             int n_rows, int topk, int32_t* indices, void* stream);

/*
 * Bytes of logits scratch that lets dsa_indexer_topk score every row in one
 * pass: total_q rows of max_seqlen_kv rounded up to 4 floats.  0 when no
 * row needs scoring (max_seqlen_kv <= topk).
 */
size_t dsa_indexer_workspace_size(int total_q, int max_seqlen_kv, int topk);

/*
 * Index lists of every query row: indices int32 [total_q, topk], written.
 * max_seqlen_kv is the longest KV sequence (total_kv for a dense sequence).
 * workspace (16-byte aligned, contents ignored) holds the logits of a chunk
 * of query rows: with less than dsa_indexer_workspace_size bytes the rows are
 * scored and selected in chunks of workspace_bytes / (4 * row length) rows
 * (the logits budget); less than one row gives
 * SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL.  The result does not depend on the
 * chunking.  Nothing is allocated; launches on `stream`.
 */
sparse_mla_status_t dsa_indexer_topk(const void* q_idx, const void* k_idx, const float* weights,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                                     int total_q, int total_kv, int max_seqlen_kv, int h_idx, int d_idx, int topk,
                                     int32_t* indices, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Decode form of the indexer over a paged key cache.  Request b has s_next
 * query rows, the last s_next of its cache_seqlens[b] positions (MTP token
 * j sits at position L_b - s_next + j and sees positions 0 .. L_b - s_next
 * + j, the convention of sparse_mla_decode); its keys live in
 *   k_cache       bf16 [num_blocks, page_size, d_idx]   16-byte aligned
 * position s of request b at row s % page_size of page
 * block_table[b * max_blocks + s / page_size] (int32 [batch, max_blocks]);
 * cache_seqlens int32 [batch].  q_idx bf16 [batch, s_next, h_idx, d_idx],
 * weights fp32 [batch, s_next, h_idx]; rows are numbered b * s_next + j.
 * page_size must be 64 (else SPARSE_MLA_ERR_UNSUPPORTED_SHAPE).  Pages past a
 * request's length are never used in a score.  A visible position whose page
 * index is at or past max_blocks, or whose page id is outside
 * [0, num_blocks), has no key: it scores -inf and is never listed (short
 * rows list only the positions that have a key).  Those are exactly the
 * positions sparse_mla_decode masks, so no listed entry is dropped by the
 * decode.  Otherwise as dsa_indexer_scores / dsa_indexer_topk (row_stride /
 * max_seqlen_kv: at least the longest cache_seqlens).
 */
sparse_mla_status_t dsa_indexer_scores_paged(const void* q_idx, const void* k_cache, const float* weights,
                                             const int32_t* block_table, const int32_t* cache_seqlens, int batch,
                                             int s_next, int h_idx, int d_idx, int page_size, int max_blocks,
                                             int num_blocks, int row0, int n_rows, int skip_len, float* scores,
                                             long long row_stride, void* stream);

sparse_mla_status_t dsa_indexer_topk_paged(const void* q_idx, const void* k_cache, const float* weights,
                                           const int32_t* block_table, const int32_t* cache_seqlens, int batch,
                                           int s_next, int h_idx, int d_idx, int page_size, int max_blocks,
                                           int num_blocks, int max_seqlen_kv, int topk, int32_t* indices,
                                           void* workspace, size_t workspace_bytes, void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* sparse_mla_status_string(sparse_mla_status_t status);

/*
 * Device error word of the current device: 0 when no kernel has timed out,
 * otherwise the code the first timed-out kernel recorded (its role in bits
 * 8..11).  Synchronises with the device.  Returns SPARSE_MLA_OK, or
 * SPARSE_MLA_ERR_CUDA if the read fails.
 */
sparse_mla_status_t sparse_mla_get_device_error(int* code);

/* Clear the current device's error word (synchronous). */
sparse_mla_status_t sparse_mla_clear_device_error(void);

/*
 * Set the bound on device-side waits, in nanoseconds, for launches made after
 * the call (process-wide; default 1 s; 0 restores the default).  Each CTA
 * restarts the clock at every unit of work it takes up (one token's head
 * group, or a CTA's share of one), so the bound applies per unit, not to the
 * whole launch.
 */
void sparse_mla_set_wait_timeout_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MLA_H */
