/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library (libattn.so).
 *
 * What is computed (the definition every entry point follows):
 *   S = scale * Q K^T,  P = softmax over each row of S restricted to the keys
 *   the mask leaves visible,  O = P V,  LSE_i = ln sum_j exp(S_ij).
 *   "DISTFLASHATTN: Distributed Memory-efficient Attention for Long-context LLMs
 *   Training" reviews, first review summary (attention = softmax(QK^T) V; the
 *   backward pass needs no recomputation of a stored N x N matrix);
 *   "FlashAttention: Fast and Memory-Efficient Exact Attention with
 *   IO-Awareness", abstract (exact attention, tiled between HBM and on-chip
 *   SRAM; block-sparse attention as the same algorithm on a block mask).
 *
 * Conventions shared by every entry point
 *   - Tensors are row-major [B, H, N, d] with d contiguous (row stride d).
 *     Q, K, V, O, dO, dQ, dK, dV are bfloat16 unless stated otherwise; LSE and
 *     D are float32 [B, H_q, N].  LSE is the natural-log log-sum-exp.
 *   - Grouped-query attention: H_q % H_kv == 0 and query head h reads key/value
 *     head h / (H_q / H_kv)  ("FlashAttention-2" reviews, first review
 *     questions: the MQA/GQA paragraph of the backward section).
 *   - d is 64 or 128.  N >= 1, any value (ragged last tiles are masked).
 *   - Every device pointer must be 16-byte aligned; head strides in bytes must
 *     be multiples of 16.
 *   - Pointers named "device" are CUDA device pointers owned by the caller; the
 *     library never frees them.  The library allocates no device memory: its
 *     status word is a static device variable, whose address on a device is
 *     looked up by that device's first call (make it before any stream
 *     capture).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *     launches are asynchronous on it.  The return value reports host-side
 *     validation and launch errors only; errors seen by a kernel are read back
 *     with attn_get_status(): a bounded wait that ran out, or a device-side
 *     index array the host cannot check (cu_seqlens, seq_lens) holding an
 *     entry out of range.
 *   - A query row that sees no key gets O = 0 and LSE = -inf.
 *   - Return codes are attn_status_t values; on error a message is available
 *     from attn_last_error_message() (thread-local) and nothing was launched.
 */
#ifndef IO_AWARE_EXACT_ATTN_GB300_ATTN_H
#define IO_AWARE_EXACT_ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1,    /* null pointer, bad size, bad mask descriptor */
  ATTN_ERR_UNSUPPORTED = -2,    /* valid but not built: d not in {64,128}, ... */
  ATTN_ERR_MISALIGNED = -3,     /* pointer or stride not 16-byte aligned */
  ATTN_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed */
  ATTN_ERR_DEVICE_TIMEOUT = -5, /* a kernel's bounded wait ran out (device-side) */
  ATTN_ERR_WORKSPACE = -6,      /* workspace too small */
  ATTN_ERR_NO_DEVICE = -7,      /* no usable sm_103 device */
  ATTN_ERR_DEVICE_BOUNDS = -8   /* a device-side index array was out of range (device-side) */
} attn_status_t;

typedef enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_BLOCK_SPARSE = 2,
  ATTN_MASK_SLIDING_WINDOW = 3
} attn_mask_kind_t;

typedef enum { ATTN_DTYPE_BF16 = 0, ATTN_DTYPE_F32 = 1 } attn_dtype_t;

/* Tile edge used by the kernels and by the block-sparse mask granularity. */
#define ATTN_TILE 128

/*
 * Mask descriptor.  A NULL attn_mask_t* means ATTN_MASK_NONE.
 *   kind = ATTN_MASK_CAUSAL: key j is visible to query i iff
 *     kv_offset + j <= q_offset + i (global positions; offsets are 0 except in
 *     attn_partial_fwd).  Fully masked key tiles are skipped, not computed
 *     ("FlashAttention-2" reviews, fourth review: causal block skipping).
 *   kind = ATTN_MASK_BLOCK_SPARSE: block_mask is a DEVICE pointer to a
 *     row-major uint8 array [ceil(Nq/128)][ceil(Nk/128)] shared by every batch
 *     and head; a nonzero byte keeps that 128x128 block dense, zero drops it
 *     and the block is skipped ("FlashAttention" abstract: block-sparse
 *     FlashAttention; BurstAttention author responses: sparse attention only
 *     changes the attention mask matrix).  causal_in_blocks != 0 additionally
 *     applies the causal rule inside kept blocks.
 *   kind = ATTN_MASK_SLIDING_WINDOW: local causal attention over the last
 *     `window` positions, the query's own included: key j is visible to query
 *     i iff 0 <= (q_offset + i) - (kv_offset + j) < window (window >= 1;
 *     "FlashAttention-2" reviews: the sliding-window attention of Mistral).
 *     Key tiles outside every row's window are skipped.
 * The descriptor is read during the call; block_mask must stay valid until the
 * launched work has completed.  window is read only for
 * ATTN_MASK_SLIDING_WINDOW.
 */
typedef struct attn_mask {
  int32_t kind;
  int32_t causal_in_blocks;
  const uint8_t* block_mask;
  int32_t window;
} attn_mask_t;

/*
 * attn_fwd -- exact attention forward with online softmax and a saved LSE.
 * "FlashAttention-2" reviews, first review questions (online-softmax
 * equations, diag(l)^-1 rescaling) and second review items 1-2 (rescaling
 * deferred to the end; one log-sum-exp saved per row for the backward pass).
 *   q   device bf16 [B, Hq,  N, d]      k, v device bf16 [B, Hkv, N, d]
 *   o   device bf16 [B, Hq,  N, d]      (written)
 *   lse device f32  [B, Hq,  N]         (written; may be NULL if not wanted)
 *   scale  multiplies Q K^T (typically 1/sqrt(d)).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int Hq, int Hkv, int N, int d, float scale,
             const attn_mask_t* mask, void* stream);

/*
 * attn_partial_fwd -- attention of one query chunk against one key/value chunk,
 * the building block of chunked / sequence-parallel attention
 * ("DISTFLASHATTN" reviews, first review summary: attention computed in chunks
 * distributed over workers; BurstAttention author responses: local attention
 * per device combined with online softmax).
 *   q        device bf16, Nq rows per head, consecutive heads q_head_stride
 *            rows apart (0 means Nq).  Layout [B, Hq, *, d].
 *   k, v     device bf16, Nk rows per head, heads kv_head_stride rows apart
 *            (0 means Nk).  Layout [B, Hkv, *, d].
 *   o_part   device f32 [B, Hq, Nq, d] contiguous: O of this chunk pair,
 *            normalised over the chunk's visible keys (0 for rows seeing none).
 *   lse_part device f32 [B, Hq, Nq]: LSE over the chunk's keys (-inf if none).
 *   q_offset, kv_offset: global positions of local row 0 / key 0, used by the
 *            causal rule.  A block-sparse mask is indexed by local tiles.
 */
int attn_partial_fwd(const void* q, const void* k, const void* v, float* o_part,
                     float* lse_part, int B, int Hq, int Hkv, int Nq, int Nk,
                     int d, float scale, const attn_mask_t* mask,
                     int64_t q_offset, int64_t kv_offset,
                     int64_t q_head_stride, int64_t kv_head_stride,
                     void* stream);

/*
 * attn_merge_lse -- combine partial results over disjoint key sets:
 *   LSE = ln sum_c exp(LSE_c),  O = sum_c exp(LSE_c - LSE) * O_c.
 * Parts with LSE_c = -inf weigh zero; a row where all parts are -inf gets
 * O = 0, LSE = -inf.  (BurstAttention author responses: online-softmax
 * combination of local results across devices.)
 *   o_parts   HOST array of n_parts DEVICE pointers, each f32 [B, Hq, Nq, d]
 *             contiguous.   lse_parts: HOST array of n_parts DEVICE pointers,
 *             each f32 [B, Hq, Nq].  1 <= n_parts <= 64.
 *   o_out     device, out_dtype (ATTN_DTYPE_BF16 or ATTN_DTYPE_F32), heads
 *             out_head_stride rows apart (0 means Nq), row stride d.
 *   lse_out   device f32, heads out_head_stride rows apart; may be NULL.
 * The pointer arrays are copied during the call.
 */
int attn_merge_lse(const float* const* o_parts, const float* const* lse_parts,
                   int n_parts, void* o_out, int out_dtype, float* lse_out,
                   int B, int Hq, int Nq, int d, int64_t out_head_stride,
                   void* stream);

/*
 * attn_bwd -- exact backward pass that recomputes P from the saved LSE instead
 * of storing it ("DISTFLASHATTN" reviews, first review point 3: the backward
 * pass needs no recomputed forward; "FlashAttention-2" reviews, second review
 * items 2-3: LSE saved for the backward pass, query-derivative update
 * restructured).  Three launches on `stream`:
 *   1. D = rowsum(dO * O) and LSE * log2 e per query row (float32, and as
 *      the dK/dV kernel's bf16 statistics operand; into the workspace);
 *   2. dK, dV per key tile, looping over the query tiles (and the query heads
 *      of its GQA group) that see it;
 *   3. dQ per query tile, accumulated in float32 on chip, looping over the key
 *      tiles it sees.
 *   q, o, dout  device bf16 [B, Hq, N, d];  k, v device bf16 [B, Hkv, N, d]
 *   lse         device f32 [B, Hq, N] from attn_fwd (same mask and scale)
 *   dq          device bf16 [B, Hq, N, d] (written)
 *   dk, dv      device bf16 [B, Hkv, N, d] (written; summed over GQA groups)
 *   workspace   device scratch of at least attn_bwd_workspace_bytes() bytes,
 *               16-byte aligned; its contents on entry are ignored.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o,
             const float* lse, const void* dout, void* dq, void* dk, void* dv,
             void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
             int N, int d, float scale, const attn_mask_t* mask, void* stream);

/*
 * attn_bwd_preprocess -- step 1 of the backward pass on its own, for the
 * chunked backward of attn_partial_bwd: per query row, D = rowsum(dO * O) and
 * LSE * log2(e), both float32, into the workspace ("FlashAttention-2"
 * reviews, second review items 2-3: the saved log-sum-exp is what the
 * backward pass recomputes P from).  Run it once per query chunk with the
 * MERGED O and LSE of that chunk (the output of attn_merge_lse over all of
 * the chunk's key chunks), so that every attn_partial_bwd of the chunk uses
 * the softmax normaliser over all of each row's keys.
 *   o, dout    device bf16, Nq rows per head, heads head_stride rows apart
 *              (0 means Nq): [B, Hq, *, d] row slices of longer tensors work.
 *   lse        device f32, Nq entries per head, heads head_stride apart.
 *   workspace  device, >= attn_bwd_workspace_bytes(B, Hq, Hq, Nq, d) bytes,
 *              16-byte aligned, caller-owned: D then LSE*log2 e, each a
 *              float array [B*Hq][ceil(Nq/128)*128] (rows past Nq hold 0 and
 *              +inf) rounded up to 256 bytes, then 32 bytes per row: -LSE*log2 e
 *              (-2^100 for +inf) and -D, each as three bf16 terms summing to
 *              the float32 value, laid out as the K = 16 operand the dK/dV
 *              kernel adds to its S^T and dP^T products (blocks of 128 rows,
 *              4 KB each, two 16-byte-per-row planes).
 */
int attn_bwd_preprocess(const void* o, const void* dout, const float* lse, int B, int Hq, int Nq, int d,
                        int64_t head_stride, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_partial_bwd -- the gradient terms of one (query chunk, key/value
 * chunk) pair of chunked attention, steps 2 and 3 of attn_bwd on the pair
 * ("DISTFLASHATTN" reviews, first review summary: attention and its backward
 * pass computed chunk by chunk over workers; BurstAttention author responses:
 * local results tied together by online-softmax statistics).  With the
 * merged statistics of attn_bwd_preprocess, P_ij = exp(S_ij - LSE_i) on the
 * pair's visible keys, and the pair contributes
 *   dV += P^T dO,  dK += scale (P * (dO V^T - D))^T Q,  dQ += scale (P * (dO V^T - D)) K;
 * summed over every pair these are the gradients of the whole sequence.
 *   q, dout    device bf16, Nq rows per head, heads q_head_stride rows apart
 *              (0 means Nq).
 *   k, v       device bf16, Nk rows per head, heads kv_head_stride rows apart
 *              (0 means Nk).
 *   workspace  the query chunk's attn_bwd_preprocess output (read only).
 *   dq         device f32 with q's layout (Nq rows per head, q_head_stride);
 *   dk, dv     device f32 with k's layout (Nk rows per head, kv_head_stride);
 *              dK, dV sum over the query heads of each GQA group.
 *   accumulate != 0: the terms are ADDED to dq, dk, dv (vector float
 *              reductions in global memory, so pairs that share an output may
 *              run concurrently on several streams; the summation order, and
 *              so the last bits, then varies).  accumulate == 0: the terms
 *              are stored (rows the pair does not reach get 0).
 *   q_offset, kv_offset: global positions of local query row 0 and key 0 for
 *              the causal and sliding-window rules, as in attn_partial_fwd
 *              (>= 0, |q_offset - kv_offset| <= 2^30, Nq + Nk <= 2^30); a
 *              block-sparse mask is indexed by the pair's local tiles.
 */
int attn_partial_bwd(const void* q, const void* k, const void* v, const void* dout, const void* workspace,
                     size_t workspace_bytes, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                     int d, float scale, const attn_mask_t* mask, int64_t q_offset, int64_t kv_offset,
                     int64_t q_head_stride, int64_t kv_head_stride, int accumulate, void* stream);

/*
 * attn_varlen_fwd -- attn_fwd over a batch of sequences of different lengths
 * packed back to back ("FlashAttention-2" reviews: variable-length inputs
 * without padding).  Sequence b holds tokens [cu_seqlens[b], cu_seqlens[b+1])
 * of the packed token-major tensors; positions, the causal rule and the
 * sliding window are local to each sequence, and no key of one sequence is
 * visible to a query of another.
 *   q           device bf16 [total, Hq,  d]   k, v device bf16 [total, Hkv, d]
 *   o           device bf16 [total, Hq,  d]   (written)
 *   lse         device f32  [Hq, total]       (written; may be NULL)
 *   cu_seqlens  device int32 [B + 1], non-decreasing, cu_seqlens[0] = 0 and
 *               cu_seqlens[B] = total; read by the kernel
 *   max_len     >= the longest sequence (work beyond it is not launched)
 *   mask        NULL, causal or sliding window (block-sparse: UNSUPPORTED)
 */
int attn_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* cu_seqlens, int B, int max_len, int64_t total,
                    int Hq, int Hkv, int d, float scale, const attn_mask_t* mask,
                    void* stream);

/*
 * attn_varlen_bwd -- attn_bwd for the packed batches of attn_varlen_fwd
 * (same layouts, cu_seqlens, max_len and mask; lse from attn_varlen_fwd).
 *   dout        device bf16 [total, Hq, d]
 *   dq          device bf16 [total, Hq, d]    dk, dv device bf16 [total, Hkv, d]
 *   workspace   device, >= attn_varlen_bwd_workspace_bytes(B, total, Hq)
 *               bytes, 256-byte aligned; caller-owned.  It holds the
 *               per-sequence tile-padded offsets and the per-row statistics
 *               of attn_bwd's workspace.
 * GQA: dK / dV sum over the query heads of a group, as in attn_bwd.
 */
int attn_varlen_bwd(const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dout, void* dq, void* dk, void* dv,
                    const int32_t* cu_seqlens, int B, int max_len, int64_t total,
                    int Hq, int Hkv, int d, float scale, const attn_mask_t* mask,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for attn_varlen_bwd: (B+1) ints rounded up to 256 bytes,
 * then the statistics of attn_bwd_workspace_bytes for Hq * (total + 127*B)
 * rows (two float arrays, then 32 bytes per row in whole 128-row blocks). */
size_t attn_varlen_bwd_workspace_bytes(int B, int64_t total, int Hq);

/*
 * attn_fwd_fp8 -- attn_fwd with e4m3 (fp8) Q, K and V, both products on the
 * fp8 tensor core ("FlashAttention: Fast and Memory-Efficient Exact Attention
 * with IO-Awareness", related papers, FlashAttention-3: FP8 attention).  The
 * stored codes are dequantised by per-tensor factors: the operation is
 *   O = softmax(scale * (q_descale Q8)(k_descale K8)^T) (v_descale V8)
 * with the mask of attn_fwd; O is bf16, LSE natural-log f32 as in attn_fwd.
 * The probabilities enter the second product as e4m3 (relative rounding
 * 2^-4 for weights w_j >= 2^-13 of the row max, absolute 2^-17 of it below),
 * so element by element |O_id - O_exact_id| <= sum_j e_j |v_jd| / sum_j w_j
 * with e_j = 2^-4 w_j (or 2^-17 below 2^-13), plus the bf16 rounding of O;
 * the row sums and the LSE stay fp32.
 *   q8          device e4m3 [B, Hq,  N, 128]   k8, v8 device e4m3 [B, Hkv, N, 128]
 *   o           device bf16 [B, Hq,  N, 128]   (written)
 *   lse         device f32  [B, Hq,  N]        (written; may be NULL)
 *   workspace   device, >= attn_fwd_fp8_workspace_bytes(B, Hkv, N, d) bytes,
 *               16-byte aligned; caller-owned.  It receives V^T.
 * d must be 128 (ATTN_ERR_UNSUPPORTED otherwise); descales finite and > 0.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, float q_descale, float k_descale,
                 float v_descale, void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
                 float scale, const attn_mask_t* mask, void* workspace, size_t workspace_bytes,
                 void* stream);

/* Workspace bytes for attn_fwd_fp8: V^T, B*Hkv*d*ceil(N/128)*128 bytes. */
size_t attn_fwd_fp8_workspace_bytes(int B, int Hkv, int N, int d);

/*
 * attn_decode_fwd -- one decoding step against a key/value cache, split over
 * the cache ("FlashAttention-2" reviews: splitting the KV cache amongst thread
 * blocks for inference).  Sequence b holds seq_lens[b] cached positions (Nk
 * each when seq_lens is NULL); its newest Nq positions are the queries: query
 * i sits at position seq_lens[b] - Nq + i and, with causal != 0, sees the
 * cached keys up to its own position, otherwise all of its sequence's keys.
 * The key range is cut into n_splits parts (0 picks a count that fills the
 * GPU); each part's attention is computed independently into the workspace
 * (fp32 O and LSE) and the parts are combined by the log-sum-exp merge of
 * attn_merge_lse.  The g = Hq/Hkv query heads of a kv head share its cache
 * reads: their g*Nq rows form one tile (g*Nq <= 256).
 *   q          device bf16 [B, Hq, Nq, d]
 *   k_cache    device bf16 [B, Hkv, Nk, d]   v_cache likewise
 *   seq_lens   device int32 [B] in [0, Nk], or NULL; read by the kernels
 *   o          device bf16 [B, Hq, Nq, d]   (written)
 *   lse        device f32 [B, Hq, Nq]       (written; may be NULL)
 *   workspace  device, >= attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d,
 *              n_splits) bytes, 16-byte aligned; caller-owned.
 * Rows of a sequence with no visible key get O = 0, LSE = -inf.
 * ATTN_ERR_INVALID_ARG for g*Nq > 256, Nq > Nk, n_splits outside [0, 64];
 * ATTN_ERR_WORKSPACE if the workspace is too small.
 */
int attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* seq_lens, void* o, float* lse, int B, int Hq,
                    int Hkv, int Nq, int Nk, int d, float scale, int causal,
                    int n_splits, void* workspace, size_t workspace_bytes,
                    void* stream);

/* Splits attn_decode_fwd uses for n_splits = 0 (at least one key tile each). */
int attn_decode_splits(int B, int Hkv, int Nk);

/* Workspace for attn_decode_fwd: per partial result, fp32 O and LSE of every
 * query row, each rounded up to 256 bytes.  A split leaves two partials when
 * a kv head's (Hq/Hkv)*Nq rows fit one 128-row tile and 2*n_splits <= 64
 * (the kernel's two query tiles then take alternate key tiles of the split),
 * one otherwise.  n_splits = 0 means attn_decode_splits. */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                   int n_splits);

/*
 * attn_bwd_static_scratch -- the same backward pass as attn_bwd, for callers
 * that must not allocate device memory: code running where cudaMalloc is not
 * allowed or would break a memory budget fixed up front (an allocator or
 * runtime that owns every device allocation, a pre-reserved serving process,
 * a host that has set up its memory pools before the hot loop).  It takes no
 * workspace and allocates nothing: its scratch (the per-row statistics that
 * attn_bwd keeps in its workspace) lives in a static device array of
 * ATTN_STATIC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.  The pages describe no such
 * variant; it is an integration aid only.
 *   Arguments, layouts and results are those of attn_bwd.
 *   Limit: B*Hq*ceil(N/128)*128 <= ATTN_STATIC_SCRATCH_ROWS (2^20) query
 *   rows; larger calls return ATTN_ERR_WORKSPACE and launch nothing.
 *   The first call on each device looks up the array's device address (and
 *   the status word's) with cudaGetSymbolAddress while that device is
 *   current; make that first call before any stream capture.
 *   All calls on a device share the one array: calls that may overlap on the
 *   GPU (other streams, other host threads) race and must be serialised by
 *   the caller.  Nothing in the array needs clearing: each call overwrites
 *   every entry it later reads.
 *   A kernel wait that runs out is reported by attn_get_status(), as for
 *   every other entry point (one status word per device serves them all).
 */
#define ATTN_STATIC_SCRATCH_ROWS (1 << 20)
#define ATTN_STATIC_SCRATCH_BYTES (40u << 20)
int attn_bwd_static_scratch(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk,
                            void* dv, int B, int Hq, int Hkv, int N, int d, float scale,
                            const attn_mask_t* mask, void* stream);

/* Bytes of workspace attn_bwd needs: 40 per query row, rows padded to whole
 * tiles (B*Hq*ceil(N/128)*128 rows): D and LSE*log2 e (two float arrays, each
 * rounded up to 256 bytes), then the same statistics as the dK/dV kernel's
 * 32-byte-per-row bf16 operand (see attn_bwd_preprocess). */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d);

/*
 * attn_build_schedule -- HOST-ONLY.  The forward work units in the order
 * attn_fwd / attn_partial_fwd launch them, as int32 triples
 * (b*Hq + h, query chunk of 256 rows, number of key tiles visited).
 * Heads are taken in groups of G = clamp((Hq/Hkv) * floor(64 MiB / (4*Nk*d)),
 * 1, B*Hq) consecutive (b, h) so that the group's K and V stay in L2; inside a
 * group the latest (heaviest) query chunk of every head comes first, then the
 * next, and so on (DISTFLASHATTN reviews, first review point 1: with causal
 * masking careless placement leaves processors idle).  host_block_mask is a
 * HOST copy of the block mask (only read for ATTN_MASK_BLOCK_SPARSE); window
 * is read only for ATTN_MASK_SLIDING_WINDOW.  Writes at most cap int32 values
 * to out and the number of units to *n_out; ATTN_ERR_INVALID_ARG if cap is
 * too small (n_out still set).
 */
int attn_build_schedule(int mask_kind, int causal_in_blocks,
                        const uint8_t* host_block_mask, int window, int B, int Hq, int Hkv,
                        int Nq, int Nk, int d, int64_t q_offset, int64_t kv_offset,
                        int32_t* out, size_t cap, size_t* n_out);

/*
 * attn_build_chunk_schedule -- HOST-ONLY.  Load-balanced order of the causal
 * (q-chunk, kv-chunk <= q-chunk) pairs of chunked attention, as int32 pairs.
 * Off-diagonal pairs cost 2, diagonal pairs 1; pairs sorted by (cost desc,
 * qc desc, kc asc) go to the least-loaded of n_lanes virtual lanes (lowest on
 * ties; n_lanes <= 0 means n_chunks) and are emitted lane-round-robin by
 * position ("DISTFLASHATTN" reviews: token-level workload balancing of the
 * causal chunks; the paper's own schedule is not reproduced on the page).
 */
int attn_build_chunk_schedule(int n_chunks, int n_lanes, int32_t* pairs_out,
                              size_t cap, size_t* n_out);

/*
 * attn_get_status -- synchronises `stream`, then reads and clears the current
 * device's status word.  Returns ATTN_OK; ATTN_ERR_DEVICE_BOUNDS if, since the
 * last call, a kernel met a malformed device-side index array (a sequence of
 * cu_seqlens with cu[b] < 0, cu[b+1] < cu[b], cu[b+1] > total or more than
 * max_len tokens: that sequence was skipped, its outputs left unwritten; a
 * seq_lens entry outside [0, Nk]: clamped into the cache); otherwise
 * ATTN_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out; ATTN_ERR_CUDA if
 * the synchronisation itself failed.
 */
int attn_get_status(void* stream);

/*
 * attn_set_wait_limit_ns -- upper bound, in nanoseconds, on every spin-wait in
 * the kernels launched after this call (default 2e9).  A wait that runs out
 * sets the status register, and the kernel drains and returns.  limit_ns <= 0
 * restores the default.
 */
void attn_set_wait_limit_ns(int64_t limit_ns);

/*
 * attn_debug_set_tile_counts -- debug record of the work each CTA did, for
 * checking the kernels against the schedule (which key tiles each query tile
 * visits: the causal and block-sparse tile skipping of the "FlashAttention-2"
 * reviews, fourth review, and the heaviest-first unit order).  From this call
 * on, every forward launch (attn_fwd, attn_partial_fwd, attn_varlen_fwd,
 * attn_decode_fwd) and every backward call (attn_bwd, attn_partial_bwd,
 * attn_varlen_bwd, attn_bwd_static_scratch) writes 8 int32 per CTA, CTA c at counts[8 * c], into
 * `counts`, a DEVICE array of `capacity` int32 that the caller owns and keeps
 * alive while recording is on.  Each launch writes from counts[0]; a backward
 * call writes its dK/dV kernel's records first and its dQ kernel's records
 * right after them.  CTAs that have no work (a chunk past the end of a shorter
 * sequence) write nothing.  Fields, per kernel:
 *   forward: [0] head index of the unit (b*Hq + h; decoding: b*Hkv + kv head;
 *            ragged batches: h), [1] first query row of the unit, [2] decode
 *            split, [3] first token of the unit's sequence (ragged batches),
 *            [4] key tiles loaded, [5] 0 (not recorded), [6] and [7] key
 *            tiles processed for query tile 0 and 1 of the unit.
 *   dK/dV:   [0] b*Hkv + kv head, [1] key tile, [2] 0, [3] first token of the
 *            sequence, [4] (query head, query tile) stages loaded, [5] query
 *            tiles whose dV and dK products were issued, [6] and [7] query
 *            tiles processed by each of the two elementwise warpgroups.
 *   dQ:      [0] b*Hq + h, [1] query tile, [2] 0, [3] first token of the
 *            sequence, [4] key tiles loaded, [5] dQ products issued, [6] and
 *            [7] key tiles processed by each elementwise warpgroup.
 * Launches whose records do not fit return ATTN_ERR_INVALID_ARG before that
 * kernel is launched.  counts == NULL turns recording off.  The e4m3 forward
 * writes no records.  Returns ATTN_ERR_MISALIGNED for a pointer that is not
 * 4-byte aligned.
 */
int attn_debug_set_tile_counts(int32_t* counts, int64_t capacity);

/*
 * attn_selftest_wait_timeout -- launches one small kernel that waits, with the
 * given limit, on a barrier that nothing signals, so that the bounded-wait
 * error path can be tested without faulting or hanging the GPU.  The wait
 * runs out after limit_ns; attn_get_status() then reports
 * ATTN_ERR_DEVICE_TIMEOUT.
 */
int attn_selftest_wait_timeout(int64_t limit_ns, void* stream);

/*
 * Launch tracing.  While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on the launching stream, so each
 * kernel's device time can be read back afterwards.  Kernel ids:
 */
typedef enum {
  ATTN_KERNEL_FWD = 1,            /* attn_fwd forward kernel */
  ATTN_KERNEL_PARTIAL_FWD = 2,    /* attn_partial_fwd forward kernel (f32 output) */
  ATTN_KERNEL_MERGE = 3,          /* attn_merge_lse */
  ATTN_KERNEL_BWD_PREPROCESS = 4, /* attn_bwd step 1: D and LSE*log2 e (also attn_bwd_preprocess) */
  ATTN_KERNEL_BWD_DKDV = 5,       /* attn_bwd step 2: dK, dV (also attn_partial_bwd) */
  ATTN_KERNEL_BWD_DQ = 6,         /* attn_bwd step 3: dQ (also attn_partial_bwd) */
  ATTN_KERNEL_SELFTEST = 7,       /* attn_selftest_wait_timeout */
  ATTN_KERNEL_DECODE = 8,         /* attn_decode_fwd split-KV partials (its merge is ATTN_KERNEL_MERGE) */
  ATTN_KERNEL_VARLEN_FWD = 9,     /* attn_varlen_fwd forward kernel */
  ATTN_KERNEL_FP8_TRANSPOSE_V = 10, /* attn_fwd_fp8 step 1: V -> V^T */
  ATTN_KERNEL_FP8_FWD = 11        /* attn_fwd_fp8 step 2: forward kernel */
} attn_kernel_id_t;

typedef struct attn_trace_record {
  int32_t kernel; /* attn_kernel_id_t */
  float ms;       /* device time between the two events */
} attn_trace_record_t;

/* Start recording (dropping earlier records); at most `capacity` launches are
 * kept (1 <= capacity <= 1<<20).  Tracing is process-wide. */
int attn_trace_enable(int capacity);
/* Stop recording; records already taken stay readable. */
int attn_trace_disable(void);
/* Wait for the recorded events, copy up to cap records in launch order to
 * out (HOST), set *n_out to the number recorded, and clear them.  Launches
 * beyond the capacity are counted in *n_out but not stored. */
int attn_trace_read(attn_trace_record_t* out, int cap, int* n_out);

const char* attn_status_string(int status);
const char* attn_last_error_message(void);
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IO_AWARE_EXACT_ATTN_GB300_ATTN_H */
