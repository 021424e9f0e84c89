// launch.h -- host-side launchers of the kernels (internal to libcsa.so).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace csa {

// Block compression (csa_compress, and csa_compress_ex with its extras:
// x_prev/z_prev, gamma and rope_dim > 0 each optional).
bool compress_supported(int D, int r, int S, int in_bytes, bool two);
cudaError_t launch_compress(const void* x, const void* z, const void* x_prev, const void* z_prev, const float* P,
                            const float* gamma, float eps, int rope_dim, float theta, int pos_stride,
                            int pos_offset, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap, int D,
                            int r, int S, bool fp32, void* out, int* status, cudaStream_t stream);
// The main KV (D) and indexer K (D_I) compressors of a layer in one launch,
// plus the compressed offsets: (D, D_I) in {(128, 64), (64, 32)}.
bool compress_pair_supported(int D, int D_I, int r, int S, int in_bytes);
cudaError_t launch_compress_pair(const void* x, const void* z, const float* P, void* out, int D, const void* x_i,
                                 const void* z_i, const float* P_i, void* out_i, int D_I, const int32_t* cu, int B,
                                 int T_cap, int r, int S, bool fp32, int32_t* cu_cmp, int* status,
                                 cudaStream_t stream);
cudaError_t launch_compressed_offsets(const int32_t* cu, int B, int r, int32_t* cu_cmp, int* status,
                                      cudaStream_t stream);

// Indexer scoring + top-k.
bool indexer_topk_supported(int H_I, int d_I, int max_vis, int k_pad, int in_bytes);
cudaError_t launch_indexer_topk(const void* qI, const void* w, const void* kI, const int32_t* cu,
                                const int32_t* cu_cmp, int B, int T_cap, int max_vis, int H_I,
                                int d_I, int r, int topk, int k_pad, bool fp32, int32_t* idx,
                                int* status, cudaStream_t stream, const int32_t* pos0 = nullptr,
                                int cmp_rows = 0);

bool indexer_topk_tc_supported(int H_I, int d_I, int max_vis, bool fp32);
cudaError_t launch_indexer_topk_tc(const void* qI, const void* w, const void* kI, const int32_t* cu,
                                   const int32_t* cu_cmp, int B, int T_cap, int max_vis, int r, int topk, int k_pad,
                                   int32_t* idx, int* status, cudaStream_t stream, const int32_t* pos0 = nullptr,
                                int cmp_rows = 0);

// FP8 indexer: E4M3 quantisation and the tcgen05 scoring + top-k on codes.
cudaError_t launch_quantize_fp8(const void* x, int64_t rows, int cols, bool fp32, uint8_t* codes, float* scales,
                                cudaStream_t stream);
cudaError_t launch_indexer_topk_fp8(const uint8_t* qI, const float* qs, const void* w, const uint8_t* kI,
                                    const float* ks, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap,
                                    int max_vis, int r, int topk, int k_pad, int32_t* idx, int* status,
                                    cudaStream_t stream, const int32_t* pos0 = nullptr,
                                int cmp_rows = 0);

cudaError_t launch_indexer_topk_fp8_full(const uint8_t* qI, const float* qs, const void* w, const uint8_t* kI,
                                         const float* ks, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap,
                                         int max_vis, int r, int topk, int k_pad, int32_t* idx, int* status,
                                         cudaStream_t stream, const int32_t* pos0 = nullptr,
                                int cmp_rows = 0);

// Attention kinds.
enum AttnKind { kAttnCSA = 0, kAttnHCA = 1, kAttnWindow = 2 };

struct AttnArgs {
  const void* q;
  const void* k_cmp;
  const void* v_cmp;
  const void* k_raw;
  const void* v_raw;
  const int32_t* idx;
  int k_pad;
  const float* sink;
  const int32_t* cu;
  const int32_t* cu_cmp;
  int B, T_cap, H, d, r, window;
  float scale;
  void* out;
  float* lse;
  float* lse_cmp;
  int* status;
  const int32_t* pos0 = nullptr;  // optional [B]: position of each sequence's first row (context parallel)
};
cudaError_t launch_attention(AttnKind kind, const AttnArgs& a, bool fp32, cudaStream_t stream);
bool attention_ws_supported(const AttnArgs& a, bool fp32);
cudaError_t launch_attention_ws(AttnKind kind, const AttnArgs& a, cudaStream_t stream);
bool attention_tc_supported(const AttnArgs& a, bool fp32);
cudaError_t launch_attention_tc(AttnKind kind, const AttnArgs& a, cudaStream_t stream);

// Attention backward: gradients of the forward above from its saved output
// and LSE.  Key / value gradients are float32 and accumulated (zeroed by the
// launcher); with K = V (v_cmp and v_raw null) dk_* receives dK + dV.
struct AttnBwdArgs {
  const void* q;
  const void* k_cmp;
  const void* v_cmp;
  const void* k_raw;
  const void* v_raw;
  const int32_t* idx;
  int k_pad;
  const float* sink;
  const int32_t* cu;
  const int32_t* cu_cmp;
  int B, T_cap, H, d, r, window;
  int n_cmp_cap;          // rows of dk_cmp / dv_cmp to zero
  float scale;
  const void* out;
  const float* lse;
  const void* dout;
  void* dq;
  float* dk_cmp;
  float* dv_cmp;
  float* dk_raw;
  float* dv_raw;
  float* dsink;
  float* delta;           // [T_cap, H] scratch: dout . out
  int* status;
  const int32_t* pos0 = nullptr;
};
cudaError_t launch_attention_bwd(AttnKind kind, const AttnBwdArgs& a, bool fp32, cudaStream_t stream);
bool attention_bwd_tc_supported(const AttnBwdArgs& a, bool fp32);
cudaError_t launch_attention_bwd_tc(AttnKind kind, const AttnBwdArgs& a, cudaStream_t stream);

struct KLArgs {
  const void* q;
  const void* k_cmp;
  const void* qI;
  const void* w;
  const void* kI;
  const int32_t* idx;   // nullptr: dense teacher over every visible entry
  int k_pad;
  const float* lse_cmp; // optional per-head normaliser over C_t (sparse mode)
  const int32_t* cu;
  const int32_t* cu_cmp;
  int B, T_cap, H, d, H_I, d_I, r;
  float scale;
  float* kl_rows;       // [T_cap] per-query KL
  int32_t* csize;       // [T_cap] |C_t|
  float* kl_sum;
  int32_t* n_valid;
  int* status;
  float* teacher_lse = nullptr;  // optional [T_cap, H]: per-head log normaliser of the teacher over C_t
  float* student_lse = nullptr;  // optional [T_cap]: log normaliser of the indexer logits over C_t
  const int32_t* pos0 = nullptr;
  int cmp_rows = 0;              // rows of the compressed arrays (0: T_cap / r)
};
cudaError_t launch_indexer_kl(const KLArgs& a, bool fp32, cudaStream_t stream);
bool indexer_kl_dense_tc_supported(const KLArgs& a, bool fp32);
cudaError_t launch_indexer_kl_dense_tc(const KLArgs& a, cudaStream_t stream);
// tcgen05 selected-set teacher (64 x 128 heads, indexer 8 x 64, bf16, with a
// reference normaliser lse_cmp); launch_indexer_kl dispatches to it.
bool indexer_kl_sparse_tc_supported(const KLArgs& a, bool fp32);
cudaError_t launch_indexer_kl_sparse_tc(const KLArgs& a, cudaStream_t stream);
// Every row as an empty C_t (KL 0, |C_t| 0, normalisers -inf).
cudaError_t launch_kl_zero_rows(float* kl_rows, int32_t* csize, int T_cap, float* teacher_lse, int H,
                                float* student_lse, cudaStream_t stream);

// Indexer KL backward: dqI, dw (I/O dtype) and float32 dkI (zeroed by the
// launcher) for upstream gradient grad_scale; the teacher is detached.
struct KLBwdArgs {
  const void* q;
  const void* k_cmp;
  const void* qI;
  const void* w;
  const void* kI;
  const int32_t* idx;   // nullptr: dense teacher
  int k_pad;
  const float* lse_cmp; // optional per-head teacher normaliser over C_t (either mode)
  const float* student_lse;  // optional student normaliser over C_t: with lse_cmp, one pass
  const int32_t* cu;
  const int32_t* cu_cmp;
  int B, T_cap, H, d, H_I, d_I, r;
  int n_cmp_cap;        // rows of dkI to zero
  float scale, grad_scale;
  void* dqI;
  void* dw;
  float* dkI;
  int* status;
  const int32_t* pos0 = nullptr;
};
cudaError_t launch_indexer_kl_bwd(const KLBwdArgs& a, bool fp32, cudaStream_t stream);
// tcgen05 one-pass backward of the dense teacher (64 x 128 heads, indexer 8 x 64,
// bf16, both normalisers given); launch_indexer_kl_bwd dispatches to it.
bool indexer_kl_bwd_tc_supported(const KLBwdArgs& a, bool fp32);
cudaError_t launch_indexer_kl_bwd_tc(const KLBwdArgs& a, cudaStream_t stream);
// tcgen05 one-pass backward of the selected-set teacher (same shapes, both
// normalisers given, gathered 128-entry tiles); launch_indexer_kl_bwd dispatches to it.
bool indexer_kl_bwd_sparse_tc_supported(const KLBwdArgs& a, bool fp32);
cudaError_t launch_indexer_kl_bwd_sparse_tc(const KLBwdArgs& a, cudaStream_t stream);

}  // namespace csa
