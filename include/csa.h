/*
 * csa.h -- C ABI of the GB300 (sm_103a) compressed sparse attention forward.
 *
 * The library computes the forward hot path of the DeepSeek-V4 compressed
 * attention layers described on the page "DeepSeek-V4 Attention Training
 * Systems" (Megatron V4 notes):
 *   1. block compression of KV (ratio 4 overlapping for CSA, ratio 128 for HCA),
 *   2. lightning-indexer scoring of every causally visible compressed entry and
 *      a per-query top-k,
 *   3. attention over the selected (CSA) or all visible (HCA) compressed
 *      entries together with the local window of raw tokens, in one softmax,
 *   4. the indexer KL auxiliary loss over the selected or the dense visible set.
 *
 * Conventions shared by every call
 * --------------------------------
 * Packing.  Tokens of B sequences are concatenated on one row axis (THD):
 *   cu_seqlens[0..B] (int32, device) with cu_seqlens[0] = 0, non-decreasing,
 *   cu_seqlens[B] <= T_cap.  Rows [cu_seqlens[B], T_cap) are capacity padding.
 *   Nothing is compressed, attended or selected across a sequence boundary
 *   (§4 "What Varlen Means In Megatron").
 * Compression.  Sequence b of length L_b owns n_b = floor(L_b / r) compressed
 *   entries (only complete groups, §4); cu_cmp[b] = sum of earlier n_b is the
 *   first packed compressed row of sequence b (csa_compressed_offsets).  Entry j
 *   is visible to local query position t once r(j+1)-1 <= t.  Compressed
 *   arrays (kv_cmp, v_cmp, kI) are capacity buffers of floor(T_cap / r) rows:
 *   the tensor-core kernels load whole 128-row tiles and may read rows past
 *   cu_cmp[B] (their values are never used).
 * Static capacity.  Buffers are sized for a fixed capacity and all metadata is
 *   read on the device, so no call synchronises with the host (§4.1 "Static
 *   capacity versus dynamic metadata").  Calls that need a bound on one
 *   sequence's length take max_seqlen (host int, >= every L_b).
 * Memory.  Every pointer is a device pointer unless stated.  The caller owns
 *   every buffer; apart from csa_create the library never allocates or frees.
 *   Arrays are dense row-major with the innermost dimension last; every array
 *   pointer must be 16-byte aligned.
 * Streams.  Every compute call only enqueues work on `stream` and returns.
 * Data types.  CSA_BF16: bf16 activations in and out.  CSA_FP32: float32
 *   arrays in and out; inputs are rounded to bf16 on load (the tensor-core
 *   operand type), outputs are written as float32.  Positional biases, sinks,
 *   LSE and KL values are always float32.
 * Errors.  Argument problems that the host can see return a negative status
 *   before anything is enqueued.  Problems only the device can see (an index
 *   outside a query's visible entries, an inconsistent cu_seqlens, a wait that
 *   ran out) set the handle's device status word and the offending element is
 *   skipped; read it with csa_get_device_status.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct csa_handle_s* csa_handle_t;

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = -1,   /* null pointer, misalignment, bad size */
  CSA_ERR_UNSUPPORTED = -2,   /* a shape this build has no kernel for */
  CSA_ERR_WORKSPACE = -3,     /* workspace missing or too small */
  CSA_ERR_CUDA = -4,          /* a CUDA runtime call failed */
  CSA_ERR_DEVICE_TIMEOUT = -5,/* a bounded device-side wait ran out */
  CSA_ERR_DEVICE_BOUNDS = -6  /* an index or cu_seqlens value out of range */
} csa_status_t;

typedef enum { CSA_BF16 = 0, CSA_FP32 = 1 } csa_dtype_t;

/* Create a handle on `device`: records device properties and allocates one
 * int32 device status word (the only allocation the library makes).
 * Returns CSA_ERR_INVALID_ARG for a null out pointer, CSA_ERR_CUDA when the
 * device cannot be used. */
csa_status_t csa_create(int device, csa_handle_t* out);

/* Free the handle and its status word.  Null is accepted. */
csa_status_t csa_destroy(csa_handle_t handle);

/* Human-readable name of a status code (static string). */
const char* csa_status_string(int status);

/* Synchronise `stream`, read the device status word into *status (host
 * pointer) and reset it to CSA_OK.  *status is CSA_OK or the first device
 * error code raised since the last read. */
csa_status_t csa_get_device_status(csa_handle_t handle, cudaStream_t stream, int* status);

/* cu_cmp[b] = sum_{b'<b} floor(L_b' / ratio) for b = 0..B (int32, device),
 * the packed compressed-row offsets (§4, complete groups only; §5.2 packed
 * compressed buffer, sequence-major).  ratio 0 gives all zeros.
 * Also checks cu_seqlens (cu[0] = 0, non-decreasing) and raises
 * CSA_ERR_DEVICE_BOUNDS on the status word if it is not. */
csa_status_t csa_compressed_offsets(csa_handle_t handle, const int32_t* cu_seqlens, int B,
                                    int ratio, int32_t* cu_cmp, cudaStream_t stream);

/* Position offsets for context-parallel layouts (§5 contiguous CP: a rank
 * holds a contiguous range of each sequence's queries plus the raw rows just
 * left of it, and all compressed rows of the sequence after the all-gather).
 * pos0 [B] int32 (device; NULL restores the default 0) is the position, in
 * its sequence, of the first packed row of each sequence segment: the query
 * calls made with this handle afterwards (top-k, attention, KL and their
 * backwards) see entry j of sequence b once r(j+1)-1 <= (row - cu[b]) + pos0[b],
 * while the window stays within the packed rows.  cmp_rows: rows of the
 * compressed arrays the caller passes from then on (they may exceed
 * floor(T_cap / ratio) after an all-gather); max_seqlen must bound the
 * positions, (row - cu[b]) + pos0[b] < max_seqlen.  The compressor is not
 * affected.  Not thread-safe with concurrent calls on the same handle. */
csa_status_t csa_set_position_offsets(csa_handle_t handle, const int32_t* pos0, int cmp_rows);

/* Learned-score block compression (§4 reset list, §5.1 spans D_compress = 8 for
 * overlapping ratio 4 and 128 for ratio-128 HCA, §8.2 "C4/C128 compression",
 * §9 FP32 compressor positional parameter).
 *   x, z      [T_cap, D]  values and gate logits (dtype)
 *   pos_bias  [S, D]      float32, S = 2*ratio (overlap = 1) or ratio
 *   out       [cu_cmp[B], D] (dtype)
 * Entry j of sequence b covers local tokens first .. first+S-1 with
 * first = ratio*j + ratio - S; per channel c,
 *   out[j,c] = sum_u softmax_u(z[t_u,c] + pos_bias[u,c]) * x[t_u,c]
 * over the span positions u with t_u >= 0 (positions before the sequence start
 * are left out).  The math is float32.  Rows of `out` past cu_cmp[B] are not
 * written.  D in {32, 64, 128, 256, 512}, ratio in 1..128, S <= 256; a span
 * whose staging rows do not fit shared memory (ratio-128 spans at D = 512)
 * returns CSA_ERR_UNSUPPORTED. */
csa_status_t csa_compress(csa_handle_t handle, const void* x, const void* z,
                          const float* pos_bias, const int32_t* cu_seqlens,
                          const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int D,
                          int ratio, int overlap, csa_dtype_t dtype, void* out,
                          cudaStream_t stream);

/* The two compressors of a CSA layer -- main KV and indexer K (§3: the
 * indexer has its own compressor; §4: both reset at packed-sample
 * boundaries) -- and their compressed offsets in one launch: the same results
 * as csa_compressed_offsets followed by csa_compress for each stream, with
 * one set of cu_seqlens, ratio and overlap.
 *   x_kv, z_kv [T_cap, D], pos_bias_kv [S, D] -> kv_cmp [cu_cmp[B], D]
 *   x_I,  z_I  [T_cap, d_I], pos_bias_I [S, d_I] -> kI_cmp [cu_cmp[B], d_I]
 *   cu_cmp [B + 1] int32, written
 * (D, d_I) must be (128, 64) or (64, 32) (CSA_ERR_UNSUPPORTED otherwise);
 * other arguments and errors as csa_compress.  No counterpart call is named
 * by the page: it fuses three of the calls above into one launch. */
csa_status_t csa_compress_pair(csa_handle_t handle, const void* x_kv, const void* z_kv,
                               const float* pos_bias_kv, const void* x_I, const void* z_I,
                               const float* pos_bias_I, const int32_t* cu_seqlens, int B, int T_cap,
                               int max_seqlen, int D, int d_I, int ratio, int overlap,
                               csa_dtype_t dtype, int32_t* cu_cmp, void* kv_cmp, void* kI_cmp,
                               cudaStream_t stream);

/* Compressor variant: csa_compress with the extras that sit around the
 * compressor in a DeepSeek-V4 layer, fused before the single rounding of the
 * output (§10 "compressor softmax and normalization intermediates"; §12
 * invariants 2 "RoPE mode is per layer and per compressed coordinate system"
 * and 3 "packed sample boundaries must reset both compressors"; §9 FP32
 * positional parameter).  Per compressed entry, in this order:
 *   1. gate     out[j,c] as csa_compress, except that with x_prev/z_prev given
 *               (overlap = 1 only) span positions u < ratio -- the previous
 *               block -- read x_prev/z_prev and u >= ratio read x/z;
 *   2. RMSNorm  (norm_weight non-null) y <- y / sqrt(mean_c y_c^2 + norm_eps)
 *               * norm_weight[c];
 *   3. RoPE     (rope_dim > 0) the trailing rope_dim channels as interleaved
 *               pairs (2i, 2i+1) rotated by p * rope_theta^(-2i/rope_dim),
 *               p = j * rope_pos_stride + rope_pos_offset with j the entry's
 *               index within its own sequence (1, 0: compressed coordinates;
 *               ratio, 0: the first token of the entry's block).
 *   x, z, x_prev, z_prev  [T_cap, D]  (dtype); x_prev, z_prev both null or both set
 *   pos_bias              [S, D]      float32
 *   norm_weight           [D]         float32 or null
 *   out                   [cu_cmp[B], D] (dtype)
 * The math is float32 (the rotation angle is reduced exactly in turns).
 * Errors: CSA_ERR_INVALID_ARG for one-sided x_prev/z_prev, x_prev without
 * overlap, an odd or oversize rope_dim, rope_theta <= 1 with rope_dim > 0 or a
 * negative norm_eps; CSA_ERR_UNSUPPORTED unless D is a power of two in
 * 32..512 and the staging rows fit shared memory (ratio-128 spans at D = 512
 * do not).  No counterpart call is named by the page: it describes these
 * steps only as parts of the layer around the compressor. */
csa_status_t csa_compress_ex(csa_handle_t handle, const void* x, const void* z, const void* x_prev,
                             const void* z_prev, const float* pos_bias, const float* norm_weight,
                             float norm_eps, int rope_dim, float rope_theta, int rope_pos_stride,
                             int rope_pos_offset, const int32_t* cu_seqlens, const int32_t* cu_cmp,
                             int B, int T_cap, int max_seqlen, int D, int ratio, int overlap,
                             csa_dtype_t dtype, void* out, cudaStream_t stream);

/* Lightning-indexer scoring and per-query top-k (§3 indexer logit i_{t,j},
 * §8 "indexer scoring and radix top-k", §8.1 top-k padding, §8.2 flat global
 * index list).  For every packed query row t of sequence b:
 *   i_{t,j} = sum_h w[t,h] * ReLU(qI[t,h,:] . kI[cu_cmp[b]+j,:]),  j < |V_t|
 * and idx[t, 0..m) holds the m = min(topk, |V_t|) entries with the largest
 * i_{t,j} (ties: smaller j first) as global compressed rows cu_cmp[b]+j in
 * ascending order; idx[t, m..k_pad) = -1.  Capacity rows get all -1.
 * Scores stay in shared memory; nothing but idx is written.
 *   qI [T_cap, H_I, d_I], w [T_cap, H_I], kI [cu_cmp[B], d_I]   (dtype)
 *   idx [T_cap, k_pad] int32
 * H_I in {1,2,4,8}, d_I in {32,64}, 1 <= topk <= k_pad <= 8192, ratio >= 1,
 * max_seqlen / ratio <= 16384. */
csa_status_t csa_indexer_topk(csa_handle_t handle, const void* qI, const void* w,
                              const void* kI, const int32_t* cu_seqlens,
                              const int32_t* cu_cmp, int B, int T_cap, int max_seqlen,
                              int H_I, int d_I, int ratio, int topk, int k_pad,
                              csa_dtype_t dtype, int32_t* idx, cudaStream_t stream);

/* FP8 indexer (§1 and §9: FP8 q^I / k^I for the index-search term; the pages
 * fix no format).  csa_quantize_fp8 turns x [rows, cols] (dtype, cols <= 256)
 * into E4M3 codes [rows, cols] (uint8) with one power-of-two scale per row
 * (float32 [rows]): s = 2^e the smallest with max|x| / s <= 448 (decided on
 * max|x| / 448 in float32; s = 1 for a zero row) and code = E4M3(x / s)
 * rounded to nearest even.  Quantise qI as [T_cap * H_I, d_I] rows and the
 * compressed indexer keys kI as [rows, d_I]. */
csa_status_t csa_quantize_fp8(csa_handle_t handle, const void* x, int64_t rows, int cols,
                              csa_dtype_t dtype, uint8_t* codes, float* scales,
                              cudaStream_t stream);

/* csa_indexer_topk on FP8 operands: qI codes [T_cap, H_I, d_I] with scales
 * qI_scale [T_cap, H_I], kI codes [., d_I] with scales kI_scale [.] (from
 * csa_quantize_fp8), w [T_cap, H_I] (bf16).  The indexer logit is that of the
 * dequantised operands,
 *   i_{t,j} = sum_h w[t,h] ReLU(qI_scale[t,h] kI_scale[j] sum_c qI[t,h,c] kI[j,c]),
 * the dot of codes on the tensor cores (E4M3 x E4M3, fp32 accumulation);
 * selection, ties, output and padding as csa_indexer_topk.  H_I = 8,
 * d_I = 64, dtype CSA_BF16 (for w) only; CSA_ERR_UNSUPPORTED otherwise. */
csa_status_t csa_indexer_topk_fp8(csa_handle_t handle, const uint8_t* qI, const float* qI_scale,
                                  const void* w, const uint8_t* kI, const float* kI_scale,
                                  const int32_t* cu_seqlens, const int32_t* cu_cmp, int B,
                                  int T_cap, int max_seqlen, int H_I, int d_I, int ratio, int topk,
                                  int k_pad, csa_dtype_t dtype, int32_t* idx, cudaStream_t stream);

/* Selected-entry attention forward, CSA (§2 phase table "top-k compressed
 * entries + local window", §8.2 selected MQA attention returning output and
 * LSE, compressed ids combined with window ids, §9 FP32 attention sink).
 * One shared KV head; for query row t of sequence b and head h the candidate
 * keys are the valid entries of idx[t,:] (global compressed rows; -1 skipped)
 * followed by the window rows cu[b]+s, s in [max(0, t-window+1), t].
 *   s_i = softmax_scale * q[t,h,:] . K_i
 *   out[t,h,:] = sum_i softmax_i(s_i; sink_h) V_i,  lse[t,h] = log(sum_i e^{s_i} + e^{sink_h})
 *   lse_cmp[t,h] = logsumexp of s_i over the compressed candidates only (no
 *   window, no sink), -inf when there are none.
 * The weights e^{s_i - m} enter the value products on the tensor cores
 * rounded to bf16 (relative error up to 2^-9), and the normalisers in lse,
 * lse_cmp and the output are the sums of those same rounded weights, so out
 * is a convex combination of the value rows with exactly the weights used
 * and out, lse combine consistently (merging partial results by their LSEs).
 * lse and lse_cmp therefore differ from the float64 log-sum-exp by up to
 * about 2e-3 when one key dominates (much less when the weight is spread).
 *   q [T_cap, H, d], kv_cmp [., d], kv_raw [T_cap, d]          (dtype)
 *   v_cmp / v_raw: separate value rows, or NULL for K = V
 *   sink [H] float32 or NULL; lse [T_cap, H], lse_cmp [T_cap, H] or NULL (float32)
 * Capacity rows: out = 0, lse = lse_cmp = -inf.  An idx entry outside the
 * query's visible entries raises CSA_ERR_DEVICE_BOUNDS and is skipped.
 * d in {64, 128}, H in {4, 8, 16, 32, 64, 128}, window >= 1, ratio >= 1. */
csa_status_t csa_sparse_attn_fwd(csa_handle_t handle, const void* q, const void* kv_cmp,
                                 const void* v_cmp, const void* kv_raw, const void* v_raw,
                                 const int32_t* idx, int k_pad, const float* sink,
                                 const int32_t* cu_seqlens, const int32_t* cu_cmp, int B,
                                 int T_cap, int max_seqlen, int H, int d, int ratio, int window,
                                 float softmax_scale, csa_dtype_t dtype, void* out, float* lse,
                                 float* lse_cmp, cudaStream_t stream);

/* HCA attention forward (§2 "HCA has no indexer: it always reads every
 * completed ratio-128 compressed entry plus the local window", §5.3).  As
 * csa_sparse_attn_fwd with the compressed candidates = every visible entry
 * cu_cmp[b] .. cu_cmp[b]+|V_t|-1.  Same layouts, limits and outputs. */
csa_status_t hca_attn_fwd(csa_handle_t handle, const void* q, const void* kv_cmp,
                          const void* v_cmp, const void* kv_raw, const void* v_raw,
                          const float* sink, const int32_t* cu_seqlens, const int32_t* cu_cmp,
                          int B, int T_cap, int max_seqlen, int H, int d, int ratio, int window,
                          float softmax_scale, csa_dtype_t dtype, void* out, float* lse,
                          float* lse_cmp, cudaStream_t stream);

/* Window-only attention forward (ratio 0 layers: no compressor, no indexer;
 * §2, §5.3).  Candidate keys are the window rows only.  lse_cmp is not
 * produced.  Same layouts and limits as csa_sparse_attn_fwd. */
csa_status_t window_attn_fwd(csa_handle_t handle, const void* q, const void* kv_raw,
                             const void* v_raw, const float* sink, const int32_t* cu_seqlens,
                             int B, int T_cap, int max_seqlen, int H, int d, int window,
                             float softmax_scale, csa_dtype_t dtype, void* out, float* lse,
                             cudaStream_t stream);

/* csa_indexer_kl that also writes the two log normalisers the indexer backward
 * needs (the page runs that backward eagerly with the forward, §8.2):
 * teacher_lse [T_cap, H] = log sum_{j in C_t} exp(softmax_scale q[t,h,:].kv_cmp[j,:])
 * and student_lse [T_cap] = log sum_{j in C_t} exp(i_{t,j}), natural units,
 * float32, -inf for capacity rows and rows with an empty C_t.  Either may be
 * NULL.  Other arguments and results as csa_indexer_kl. */
csa_status_t csa_indexer_kl_ex(csa_handle_t handle, const void* q, const void* kv_cmp,
                               const void* qI, const void* w, const void* kI, const int32_t* idx,
                               int k_pad, const float* lse_cmp, const int32_t* cu_seqlens,
                               const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H,
                               int d, int H_I, int d_I, int ratio, float softmax_scale,
                               csa_dtype_t dtype, float* kl_sum, float* kl_per_query,
                               int32_t* n_valid, void* ws, size_t ws_bytes, float* teacher_lse,
                               float* student_lse, cudaStream_t stream);

/* Attention backward, CSA (§8.2 "main attention backward": consumes the saved
 * output and LSE and produces Q, KV and attention-sink gradients without
 * materializing a dense attention matrix; §9 FP32 sink and softmax math).
 * Arguments up to `dtype` are those of the forward call whose gradient is
 * taken; out and lse are that call's outputs (out in dtype, lse float32).
 * Given dout = dL/dout [T_cap, H, d] (dtype), with p_i = exp(s_i - lse[t,h]):
 *   D[t,h]      = dout[t,h,:] . out[t,h,:]            (written to delta)
 *   ds_i        = p_i (dout[t,h,:] . V_i - D[t,h])
 *   dq[t,h,:]   = softmax_scale sum_i ds_i K_i          (dtype; capacity rows 0)
 *   dK_i       += softmax_scale ds_i q[t,h,:],   dV_i += p_i dout[t,h,:]
 *   dsink[h]    = -sum_t exp(sink[h] - lse[t,h]) D[t,h]
 * Key / value gradients are float32 and summed over every query and head:
 *   dkv_cmp [floor(T_cap/ratio), d], dkv_raw [T_cap, d]  receive dK (+ dV when
 *   K = V, i.e. v_cmp / v_raw NULL: the gradient of the shared KV rows);
 *   dv_cmp, dv_raw receive dV when V is separate, NULL otherwise.
 * The call zeroes them first; the sums are float32 atomic additions, so
 * their low bits depend on the order the GPU runs them in.  dsink [H] is
 * written when both sink and dsink are given.  delta [T_cap, H] float32 is
 * scratch (D above).  Errors as the forward; in addition every gradient
 * array must be 16-byte aligned and dv_* set exactly when V is separate. */
csa_status_t csa_sparse_attn_bwd(csa_handle_t handle, const void* q, const void* kv_cmp,
                                 const void* v_cmp, const void* kv_raw, const void* v_raw,
                                 const int32_t* idx, int k_pad, const float* sink,
                                 const int32_t* cu_seqlens, const int32_t* cu_cmp, int B,
                                 int T_cap, int max_seqlen, int H, int d, int ratio, int window,
                                 float softmax_scale, csa_dtype_t dtype, const void* out,
                                 const float* lse, const void* dout, void* dq, float* dkv_cmp,
                                 float* dv_cmp, float* dkv_raw, float* dv_raw, float* dsink,
                                 float* delta, cudaStream_t stream);

/* HCA attention backward: as csa_sparse_attn_bwd with the compressed
 * candidates of hca_attn_fwd (every visible entry). */
csa_status_t hca_attn_bwd(csa_handle_t handle, const void* q, const void* kv_cmp,
                          const void* v_cmp, const void* kv_raw, const void* v_raw,
                          const float* sink, const int32_t* cu_seqlens, const int32_t* cu_cmp,
                          int B, int T_cap, int max_seqlen, int H, int d, int ratio, int window,
                          float softmax_scale, csa_dtype_t dtype, const void* out,
                          const float* lse, const void* dout, void* dq, float* dkv_cmp,
                          float* dv_cmp, float* dkv_raw, float* dv_raw, float* dsink,
                          float* delta, cudaStream_t stream);

/* Window-only attention backward: as csa_sparse_attn_bwd with the window rows
 * as the only candidates (no compressed gradients). */
csa_status_t window_attn_bwd(csa_handle_t handle, const void* q, const void* kv_raw,
                             const void* v_raw, const float* sink, const int32_t* cu_seqlens,
                             int B, int T_cap, int max_seqlen, int H, int d, int window,
                             float softmax_scale, csa_dtype_t dtype, const void* out,
                             const float* lse, const void* dout, void* dq, float* dkv_raw,
                             float* dv_raw, float* dsink, float* delta, cudaStream_t stream);

/* Indexer KL auxiliary loss (§3 equation
 *   L_I = sum_t KL(Softmax(a_{t,C_t}) || Softmax(i_{t,C_t})),
 * §2 phase table: dense teacher over every visible entry in the sparse
 * warm-up, selected-set teacher in sparse mode; §9 FP32 loss math).
 *   C_t     = valid entries of idx[t,:] (idx != NULL) or every visible entry
 *   pi_h(j) = softmax over C_t of softmax_scale * q[t,h,:] . kv_cmp[j,:]
 *   p(j)    = (1/H) sum_h pi_h(j)          (teacher; a_{t,j} = log p(j))
 *   q(j)    = softmax over C_t of i_{t,j}  (indexer logits as in csa_indexer_topk)
 *   kl_per_query[t] = sum_j p(j) (log p(j) - log q(j)), 0 when C_t is empty
 *   kl_sum[0]  = sum over rows of kl_per_query (float32, fixed summation order)
 *   n_valid[0] = number of rows with a non-empty C_t
 * lse_cmp (sparse mode only, may be NULL): a reference for the teacher's
 * per-head log normaliser over C_t, within a few units of it --
 * csa_sparse_attn_fwd's lse_cmp is one.  The teacher's exact normaliser is
 * computed either way (a first pass over C_t); with the reference, 64 heads x
 * 128 and an 8 x 64 indexer in bf16 run on the tensor cores, the first pass
 * summing exp(s - reference) per head.  A reference more than about 22 below
 * the true value raises CSA_ERR_DEVICE_BOUNDS.  kl_per_query and n_valid may
 * be NULL.
 * ws/ws_bytes: device scratch of at least csa_indexer_kl_workspace(T_cap)
 * bytes (per-query partial results); CSA_ERR_WORKSPACE otherwise.
 * Same layouts as csa_indexer_topk / csa_sparse_attn_fwd. */
csa_status_t csa_indexer_kl(csa_handle_t handle, const void* q, const void* kv_cmp,
                            const void* qI, const void* w, const void* kI, const int32_t* idx,
                            int k_pad, const float* lse_cmp, const int32_t* cu_seqlens,
                            const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H,
                            int d, int H_I, int d_I, int ratio, float softmax_scale,
                            csa_dtype_t dtype, float* kl_sum, float* kl_per_query,
                            int32_t* n_valid, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Scratch bytes csa_indexer_kl needs for T_cap packed rows. */
size_t csa_indexer_kl_workspace(int T_cap);

/* csa_indexer_kl for callers that cannot allocate device memory (no
 * counterpart on the page: it is a deployment convenience).  Some callers
 * cannot provide a workspace -- code whose device memory is owned entirely by
 * a host framework or captured into a graph it does not control, processes
 * that forbid allocations after start-up.  This variant takes the same
 * arguments minus ws/ws_bytes and uses a fixed 2 MiB scratch array that lives
 * in the library's device image (held on every GPU that loads the library
 * until the process exits).  It makes no allocation of any kind.
 *   - T_cap must be <= 262144; larger returns CSA_ERR_WORKSPACE.
 *   - The first call on each device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *     The address is kept for the life of the process: after a
 *     cudaDeviceReset (or any other teardown of the device's primary
 *     context) it is stale, and this entry point must not be called again on
 *     that device in the same process.
 *   - Calls share the array: calls that overlap on the GPU race on it, so the
 *     caller serialises them.  Each call writes every scratch element it
 *     reads, so leftover contents from an earlier call are never used.
 * Results are identical to csa_indexer_kl with a caller workspace. */
csa_status_t csa_indexer_kl_static_scratch(csa_handle_t handle, const void* q, const void* kv_cmp,
                                           const void* qI, const void* w, const void* kI,
                                           const int32_t* idx, int k_pad, const float* lse_cmp,
                                           const int32_t* cu_seqlens, const int32_t* cu_cmp, int B,
                                           int T_cap, int max_seqlen, int H, int d, int H_I, int d_I,
                                           int ratio, float softmax_scale, csa_dtype_t dtype,
                                           float* kl_sum, float* kl_per_query, int32_t* n_valid,
                                           cudaStream_t stream);

/* Indexer backward: gradients of the indexer KL loss of csa_indexer_kl with
 * respect to the indexer inputs (§8.2 "indexer backward": the discrete top-k
 * has no LM-loss gradient, so the indexer learns through this auxiliary loss
 * only; the teacher operands q and kv_cmp are detached).  With p(j), q(j) and
 * C_t as in csa_indexer_kl and a_{h,j} = qI[t,h,:] . kI[j,:]:
 *   g_j          = grad_scale * (q(j) - p(j))            (dL_I / d i_{t,j})
 *   dw[t,h]      = sum_{j in C_t} g_j ReLU(a_{h,j})
 *   dqI[t,h,:]   = w[t,h] sum_{j in C_t} g_j [a_{h,j} > 0] kI[j,:]
 *   dkI[j,:]    += sum_t sum_h g_j w[t,h] [a_{h,j} > 0] qI[t,h,:]
 * grad_scale is the upstream gradient of L_I (1 for the unit gradient the page
 * uses when it runs this step eagerly inside the forward; the loss scale can
 * be passed here or applied later).  dqI [T_cap, H_I, d_I] and dw [T_cap, H_I]
 * (dtype) are written (0 for capacity rows and rows with an empty C_t); dkI
 * [floor(T_cap/ratio), d_I] float32 is zeroed and accumulated with float32
 * atomic additions.  idx as in csa_indexer_kl.  lse_cmp (may be NULL): the
 * teacher's per-head log normaliser over C_t -- the teacher_lse of
 * csa_indexer_kl_ex (csa_sparse_attn_fwd's lse_cmp is that of its
 * bf16-rounded weights, within about 2e-3 of it);
 * student_lse (may be NULL): the student's, from csa_indexer_kl_ex.  With both
 * the call takes one pass over C_t instead of two (for the dense teacher at 64
 * heads x 128 and an 8 x 64 indexer in bf16, on the tensor cores).  dqI and dw
 * are deterministic; dkI's float32 sums follow the order of the atomic
 * additions and may differ in the last bits between runs.  Same limits. */
csa_status_t csa_indexer_kl_bwd(csa_handle_t handle, const void* q, const void* kv_cmp,
                                const void* qI, const void* w, const void* kI, const int32_t* idx,
                                int k_pad, const float* lse_cmp, const float* student_lse,
                                const int32_t* cu_seqlens,
                                const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H,
                                int d, int H_I, int d_I, int ratio, float softmax_scale,
                                float grad_scale, csa_dtype_t dtype, void* dqI, void* dw,
                                float* dkI, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
