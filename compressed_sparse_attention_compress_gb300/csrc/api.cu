// api.cu -- the extern "C" boundary of libcsa.so: handle, argument checks,
// dispatch to the kernels.  Declarations and the contract are in include/csa.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "../../include/csa.h"
#include "launch.h"

struct csa_handle_s {
  int device;
  int sm_count;
  int* status;               // one int32 device word
  const int32_t* pos0;       // per-sequence position of the first row (csa_set_position_offsets), or null
  int cmp_rows;              // rows of the compressed arrays when pos0 is set (0: T_cap / ratio)
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Null or 16-byte aligned (optional arguments).
bool opt_aligned16(const void* p) { return p == nullptr || aligned16(p); }

csa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

// Shared checks of the packing arguments.
bool packing_ok(const int32_t* cu, int B, int T_cap, int max_seqlen) {
  return cu != nullptr && B >= 0 && T_cap >= 0 && max_seqlen >= 0 && (B == 0 || max_seqlen >= 1);
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" {

csa_status_t csa_create(int device, csa_handle_t* out) {
  if (out == nullptr) return CSA_ERR_INVALID_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) return CSA_ERR_CUDA;
  DeviceGuard g(device);
  if (!g.ok) return CSA_ERR_CUDA;
  csa_handle_s* h = static_cast<csa_handle_s*>(calloc(1, sizeof(csa_handle_s)));
  if (!h) return CSA_ERR_CUDA;
  h->device = device;
  if (cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaMalloc(&h->status, sizeof(int)) != cudaSuccess || cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) {
    if (h->status) cudaFree(h->status);
    free(h);
    return CSA_ERR_CUDA;
  }
  *out = h;
  return CSA_OK;
}

csa_status_t csa_destroy(csa_handle_t h) {
  if (!h) return CSA_OK;
  DeviceGuard g(h->device);
  cudaFree(h->status);
  free(h);
  return CSA_OK;
}

const char* csa_status_string(int s) {
  switch (s) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_INVALID_ARG: return "CSA_ERR_INVALID_ARG";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED";
    case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA";
    case CSA_ERR_DEVICE_TIMEOUT: return "CSA_ERR_DEVICE_TIMEOUT";
    case CSA_ERR_DEVICE_BOUNDS: return "CSA_ERR_DEVICE_BOUNDS";
    default: return "CSA_UNKNOWN_STATUS";
  }
}

csa_status_t csa_set_position_offsets(csa_handle_t h, const int32_t* pos0, int cmp_rows) {
  if (!h || cmp_rows < 0 || (pos0 != nullptr && (reinterpret_cast<uintptr_t>(pos0) & 3u) != 0))
    return CSA_ERR_INVALID_ARG;
  h->pos0 = pos0;
  h->cmp_rows = pos0 != nullptr ? cmp_rows : 0;
  return CSA_OK;
}

csa_status_t csa_get_device_status(csa_handle_t h, cudaStream_t stream, int* status) {
  if (!h || !status) return CSA_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  int v = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA_ERR_CUDA;
  if (cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
  if (cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) return CSA_ERR_CUDA;
  *status = v;
  return CSA_OK;
}

csa_status_t csa_compressed_offsets(csa_handle_t h, const int32_t* cu, int B, int ratio, int32_t* cu_cmp,
                                    cudaStream_t stream) {
  if (!h || !cu || !cu_cmp || B < 0 || ratio < 0) return CSA_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  return from_cuda(csa::launch_compressed_offsets(cu, B, ratio, cu_cmp, h->status, stream));
}

csa_status_t csa_compress(csa_handle_t h, const void* x, const void* z, const float* pos_bias,
                          const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int D,
                          int ratio, int overlap, csa_dtype_t dtype, void* out, cudaStream_t stream) {
  if (!h || !x || !z || !pos_bias || !cu_cmp || !out || !packing_ok(cu, B, T_cap, max_seqlen))
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(z) || !aligned16(out) || !aligned16(pos_bias)) return CSA_ERR_INVALID_ARG;
  if ((dtype != CSA_BF16 && dtype != CSA_FP32) || (overlap != 0 && overlap != 1) || ratio < 1)
    return CSA_ERR_INVALID_ARG;
  const int S = overlap ? 2 * ratio : ratio;
  if (!pow2_in(D, 32, 512) || ratio > 128 || S > 256) return CSA_ERR_UNSUPPORTED;
  const bool fp32 = dtype == CSA_FP32;
  if (!csa::compress_supported(D, ratio, S, fp32 ? 4 : 2, false)) return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  return from_cuda(csa::launch_compress(x, z, nullptr, nullptr, pos_bias, nullptr, 0.f, 0, 0.f, 0, 0, cu, cu_cmp, B,
                                        T_cap, D, ratio, S, fp32, out, h->status, stream));
}

csa_status_t csa_compress_pair(csa_handle_t h, const void* x_kv, const void* z_kv, const float* pos_bias_kv,
                               const void* x_I, const void* z_I, const float* pos_bias_I, const int32_t* cu,
                               int B, int T_cap, int max_seqlen, int D, int d_I, int ratio, int overlap,
                               csa_dtype_t dtype, int32_t* cu_cmp, void* kv_cmp, void* kI_cmp, cudaStream_t stream) {
  if (!h || !x_kv || !z_kv || !pos_bias_kv || !x_I || !z_I || !pos_bias_I || !cu_cmp || !kv_cmp || !kI_cmp ||
      !packing_ok(cu, B, T_cap, max_seqlen))
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(x_kv) || !aligned16(z_kv) || !aligned16(pos_bias_kv) || !aligned16(x_I) || !aligned16(z_I) ||
      !aligned16(pos_bias_I) || !aligned16(kv_cmp) || !aligned16(kI_cmp))
    return CSA_ERR_INVALID_ARG;
  if ((dtype != CSA_BF16 && dtype != CSA_FP32) || (overlap != 0 && overlap != 1) || ratio < 1)
    return CSA_ERR_INVALID_ARG;
  const int S = overlap ? 2 * ratio : ratio;
  const bool fp32 = dtype == CSA_FP32;
  if (ratio > 128 || S > 256 || !csa::compress_pair_supported(D, d_I, ratio, S, fp32 ? 4 : 2))
    return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  return from_cuda(csa::launch_compress_pair(x_kv, z_kv, pos_bias_kv, kv_cmp, D, x_I, z_I, pos_bias_I, kI_cmp, d_I,
                                             cu, B, T_cap, ratio, S, fp32, cu_cmp, h->status, stream));
}

csa_status_t csa_compress_ex(csa_handle_t h, const void* x, const void* z, const void* x_prev,
                             const void* z_prev, const float* pos_bias, const float* norm_weight, float norm_eps,
                             int rope_dim, float rope_theta, int rope_pos_stride, int rope_pos_offset,
                             const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int D,
                             int ratio, int overlap, csa_dtype_t dtype, void* out, cudaStream_t stream) {
  if (!h || !x || !z || !pos_bias || !cu_cmp || !out || !packing_ok(cu, B, T_cap, max_seqlen))
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(z) || !aligned16(out) || !aligned16(pos_bias) || !opt_aligned16(x_prev) ||
      !opt_aligned16(z_prev) || !opt_aligned16(norm_weight))
    return CSA_ERR_INVALID_ARG;
  if ((dtype != CSA_BF16 && dtype != CSA_FP32) || (overlap != 0 && overlap != 1) || ratio < 1)
    return CSA_ERR_INVALID_ARG;
  const bool two = x_prev != nullptr;
  if (two != (z_prev != nullptr) || (two && !overlap)) return CSA_ERR_INVALID_ARG;
  if (rope_dim < 0 || rope_dim > D || (rope_dim & 1) || !(norm_eps >= 0.f) ||
      (rope_dim > 0 && !(rope_theta > 1.f)))
    return CSA_ERR_INVALID_ARG;
  const int S = overlap ? 2 * ratio : ratio;
  if (!pow2_in(D, 32, 512) || ratio > 128 || S > 256) return CSA_ERR_UNSUPPORTED;
  const bool fp32 = dtype == CSA_FP32;
  if (!csa::compress_supported(D, ratio, S, fp32 ? 4 : 2, two)) return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  return from_cuda(csa::launch_compress(x, z, x_prev, z_prev, pos_bias, norm_weight, norm_eps, rope_dim,
                                           rope_theta, rope_pos_stride, rope_pos_offset, cu, cu_cmp, B, T_cap, D,
                                           ratio, S, fp32, out, h->status, stream));
}

csa_status_t csa_indexer_topk(csa_handle_t h, const void* qI, const void* w, const void* kI, const int32_t* cu,
                              const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H_I, int d_I, int ratio,
                              int topk, int k_pad, csa_dtype_t dtype, int32_t* idx, cudaStream_t stream) {
  if (!h || !qI || !w || !kI || !cu_cmp || !idx || !packing_ok(cu, B, T_cap, max_seqlen))
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(qI) || !aligned16(kI) || !aligned16(idx)) return CSA_ERR_INVALID_ARG;
  if ((dtype != CSA_BF16 && dtype != CSA_FP32) || ratio < 1 || topk < 1 || k_pad < topk)
    return CSA_ERR_INVALID_ARG;
  if (!pow2_in(H_I, 1, 8) || (d_I != 32 && d_I != 64) || k_pad > 8192) return CSA_ERR_UNSUPPORTED;
  const int max_vis = max_seqlen / ratio;
  if (max_vis > 16384) return CSA_ERR_UNSUPPORTED;
  const bool fp32 = dtype == CSA_FP32;
  if (!csa::indexer_topk_supported(H_I, d_I, max_vis, k_pad, fp32 ? 4 : 2)) return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  return from_cuda(csa::launch_indexer_topk(qI, w, kI, cu, cu_cmp, B, T_cap, max_vis, H_I, d_I, ratio, topk, k_pad,
                                            fp32, idx, h->status, stream, h->pos0, h->cmp_rows));
}

static csa_status_t attn_common(csa::AttnKind kind, csa_handle_t h, const void* q, const void* kv_cmp,
                                const void* v_cmp, const void* kv_raw, const void* v_raw, const int32_t* idx,
                                int k_pad, const float* sink, const int32_t* cu, const int32_t* cu_cmp, int B,
                                int T_cap, int max_seqlen, int H, int d, int ratio, int window, float scale,
                                csa_dtype_t dtype, void* out, float* lse, float* lse_cmp, cudaStream_t stream) {
  if (!h || !q || !kv_raw || !out || !lse || !packing_ok(cu, B, T_cap, max_seqlen)) return CSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_raw) || !aligned16(out) || !opt_aligned16(v_raw) || !opt_aligned16(v_cmp))
    return CSA_ERR_INVALID_ARG;
  if (kind != csa::kAttnWindow) {
    if (!kv_cmp || !cu_cmp || !aligned16(kv_cmp) || ratio < 1) return CSA_ERR_INVALID_ARG;
    if ((v_cmp == nullptr) != (v_raw == nullptr)) return CSA_ERR_INVALID_ARG;  // both or neither
  }
  if (kind == csa::kAttnCSA && (!idx || k_pad < 1)) return CSA_ERR_INVALID_ARG;
  if ((dtype != CSA_BF16 && dtype != CSA_FP32) || window < 1 || !(scale > 0.f)) return CSA_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || !pow2_in(H, 4, 128)) return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  csa::AttnArgs a{q, kv_cmp, v_cmp, kv_raw, v_raw, idx, k_pad, sink, cu, cu_cmp, B, T_cap, H, d,
                  ratio, window, scale, out, lse, lse_cmp, h->status, h->pos0};
  return from_cuda(csa::launch_attention(kind, a, dtype == CSA_FP32, stream));
}

csa_status_t csa_sparse_attn_fwd(csa_handle_t h, const void* q, const void* kv_cmp, const void* v_cmp,
                                 const void* kv_raw, const void* v_raw, const int32_t* idx, int k_pad,
                                 const float* sink, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap,
                                 int max_seqlen, int H, int d, int ratio, int window, float scale,
                                 csa_dtype_t dtype, void* out, float* lse, float* lse_cmp, cudaStream_t stream) {
  return attn_common(csa::kAttnCSA, h, q, kv_cmp, v_cmp, kv_raw, v_raw, idx, k_pad, sink, cu, cu_cmp, B, T_cap,
                     max_seqlen, H, d, ratio, window, scale, dtype, out, lse, lse_cmp, stream);
}

csa_status_t hca_attn_fwd(csa_handle_t h, const void* q, const void* kv_cmp, const void* v_cmp,
                          const void* kv_raw, const void* v_raw, const float* sink, const int32_t* cu,
                          const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H, int d, int ratio,
                          int window, float scale, csa_dtype_t dtype, void* out, float* lse, float* lse_cmp,
                          cudaStream_t stream) {
  return attn_common(csa::kAttnHCA, h, q, kv_cmp, v_cmp, kv_raw, v_raw, nullptr, 0, sink, cu, cu_cmp, B, T_cap,
                     max_seqlen, H, d, ratio, window, scale, dtype, out, lse, lse_cmp, stream);
}

csa_status_t window_attn_fwd(csa_handle_t h, const void* q, const void* kv_raw, const void* v_raw,
                             const float* sink, const int32_t* cu, int B, int T_cap, int max_seqlen, int H, int d,
                             int window, float scale, csa_dtype_t dtype, void* out, float* lse,
                             cudaStream_t stream) {
  return attn_common(csa::kAttnWindow, h, q, nullptr, nullptr, kv_raw, v_raw, nullptr, 0, sink, cu, nullptr, B,
                     T_cap, max_seqlen, H, d, 0, window, scale, dtype, out, lse, nullptr, stream);
}

static csa_status_t attn_bwd_common(csa::AttnKind kind, csa_handle_t h, const void* q, const void* kv_cmp,
                                    const void* v_cmp, const void* kv_raw, const void* v_raw, const int32_t* idx,
                                    int k_pad, const float* sink, const int32_t* cu, const int32_t* cu_cmp, int B,
                                    int T_cap, int max_seqlen, int H, int d, int ratio, int window, float scale,
                                    csa_dtype_t dtype, const void* out, const float* lse, const void* dout,
                                    void* dq, float* dkv_cmp, float* dv_cmp, float* dkv_raw, float* dv_raw,
                                    float* dsink, float* delta, cudaStream_t stream) {
  if (!h || !q || !kv_raw || !out || !lse || !dout || !dq || !dkv_raw || !delta ||
      !packing_ok(cu, B, T_cap, max_seqlen))
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_raw) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dkv_raw) || !aligned16(lse) || !aligned16(delta) || !opt_aligned16(v_raw) ||
      !opt_aligned16(v_cmp) || !opt_aligned16(dv_cmp) || !opt_aligned16(dv_raw) || !opt_aligned16(dkv_cmp))
    return CSA_ERR_INVALID_ARG;
  if ((v_raw == nullptr) != (dv_raw == nullptr)) return CSA_ERR_INVALID_ARG;  // dV wanted iff V is separate
  if (kind != csa::kAttnWindow) {
    if (!kv_cmp || !cu_cmp || !dkv_cmp || !aligned16(kv_cmp) || ratio < 1) return CSA_ERR_INVALID_ARG;
    if ((v_cmp == nullptr) != (v_raw == nullptr) || (v_cmp == nullptr) != (dv_cmp == nullptr))
      return CSA_ERR_INVALID_ARG;
  }
  if (kind == csa::kAttnCSA && (!idx || k_pad < 1)) return CSA_ERR_INVALID_ARG;
  if ((dtype != CSA_BF16 && dtype != CSA_FP32) || window < 1 || !(scale > 0.f)) return CSA_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || !pow2_in(H, 4, 128)) return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  const int n_cmp_cap = kind == csa::kAttnWindow ? 0 : (h->cmp_rows > T_cap / ratio ? h->cmp_rows : T_cap / ratio);
  csa::AttnBwdArgs a{q, kv_cmp, v_cmp, kv_raw, v_raw, idx, k_pad, sink, cu, cu_cmp, B, T_cap, H, d,
                     kind == csa::kAttnWindow ? 0 : ratio, window, n_cmp_cap, scale, out, lse, dout, dq,
                     kind == csa::kAttnWindow ? nullptr : dkv_cmp, kind == csa::kAttnWindow ? nullptr : dv_cmp,
                     dkv_raw, dv_raw, dsink, delta, h->status, h->pos0};
  return from_cuda(csa::launch_attention_bwd(kind, a, dtype == CSA_FP32, stream));
}

csa_status_t csa_sparse_attn_bwd(csa_handle_t h, const void* q, const void* kv_cmp, const void* v_cmp,
                                 const void* kv_raw, const void* v_raw, const int32_t* idx, int k_pad,
                                 const float* sink, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap,
                                 int max_seqlen, int H, int d, int ratio, int window, float scale,
                                 csa_dtype_t dtype, const void* out, const float* lse, const void* dout, void* dq,
                                 float* dkv_cmp, float* dv_cmp, float* dkv_raw, float* dv_raw, float* dsink,
                                 float* delta, cudaStream_t stream) {
  return attn_bwd_common(csa::kAttnCSA, h, q, kv_cmp, v_cmp, kv_raw, v_raw, idx, k_pad, sink, cu, cu_cmp, B,
                         T_cap, max_seqlen, H, d, ratio, window, scale, dtype, out, lse, dout, dq, dkv_cmp,
                         dv_cmp, dkv_raw, dv_raw, dsink, delta, stream);
}

csa_status_t hca_attn_bwd(csa_handle_t h, const void* q, const void* kv_cmp, const void* v_cmp,
                          const void* kv_raw, const void* v_raw, const float* sink, const int32_t* cu,
                          const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H, int d, int ratio,
                          int window, float scale, csa_dtype_t dtype, const void* out, const float* lse,
                          const void* dout, void* dq, float* dkv_cmp, float* dv_cmp, float* dkv_raw,
                          float* dv_raw, float* dsink, float* delta, cudaStream_t stream) {
  return attn_bwd_common(csa::kAttnHCA, h, q, kv_cmp, v_cmp, kv_raw, v_raw, nullptr, 0, sink, cu, cu_cmp, B,
                         T_cap, max_seqlen, H, d, ratio, window, scale, dtype, out, lse, dout, dq, dkv_cmp,
                         dv_cmp, dkv_raw, dv_raw, dsink, delta, stream);
}

csa_status_t window_attn_bwd(csa_handle_t h, const void* q, const void* kv_raw, const void* v_raw,
                             const float* sink, const int32_t* cu, int B, int T_cap, int max_seqlen, int H, int d,
                             int window, float scale, csa_dtype_t dtype, const void* out, const float* lse,
                             const void* dout, void* dq, float* dkv_raw, float* dv_raw, float* dsink, float* delta,
                             cudaStream_t stream) {
  return attn_bwd_common(csa::kAttnWindow, h, q, nullptr, nullptr, kv_raw, v_raw, nullptr, 0, sink, cu, nullptr,
                         B, T_cap, max_seqlen, H, d, 0, window, scale, dtype, out, lse, dout, dq, nullptr, nullptr,
                         dkv_raw, dv_raw, dsink, delta, stream);
}

size_t csa_indexer_kl_workspace(int T_cap) {
  if (T_cap < 0) return 0;
  return ((size_t)T_cap * 8 + 255) & ~(size_t)255;  // float kl[T_cap] + int32 csize[T_cap]
}

static csa_status_t indexer_kl_common(csa_handle_t h, const void* q, const void* kv_cmp, const void* qI, const void* w,
                            const void* kI, const int32_t* idx, int k_pad, const float* lse_cmp, const int32_t* cu,
                            const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H, int d, int H_I,
                            int d_I, int ratio, float scale, csa_dtype_t dtype, float* kl_sum, float* kl_per_query,
                            int32_t* n_valid, void* ws, size_t ws_bytes, float* teacher_lse, float* student_lse,
                                       cudaStream_t stream) {
  if (!h || !q || !kv_cmp || !qI || !w || !kI || !cu_cmp || !kl_sum || !packing_ok(cu, B, T_cap, max_seqlen))
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cmp) || !aligned16(qI) || !aligned16(kI)) return CSA_ERR_INVALID_ARG;
  if ((dtype != CSA_BF16 && dtype != CSA_FP32) || ratio < 1 || !(scale > 0.f)) return CSA_ERR_INVALID_ARG;
  if (idx != nullptr && k_pad < 1) return CSA_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || !pow2_in(H, 4, 128) || !pow2_in(H_I, 1, 8) || (d_I != 32 && d_I != 64))
    return CSA_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < csa_indexer_kl_workspace(T_cap) || !aligned16(ws)) return CSA_ERR_WORKSPACE;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  float* kl_rows = kl_per_query ? kl_per_query : static_cast<float*>(ws);
  int32_t* csize = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + (size_t)T_cap * 4);
  if (!opt_aligned16(teacher_lse) || !opt_aligned16(student_lse)) return CSA_ERR_INVALID_ARG;
  csa::KLArgs a{q, kv_cmp, qI, w, kI, idx, k_pad, lse_cmp, cu, cu_cmp, B, T_cap, H, d, H_I, d_I, ratio,
                scale, kl_rows, csize, kl_sum, n_valid, h->status, teacher_lse, student_lse, h->pos0, h->cmp_rows};
  return from_cuda(csa::launch_indexer_kl(a, dtype == CSA_FP32, stream));
}

csa_status_t csa_indexer_kl(csa_handle_t h, const void* q, const void* kv_cmp, const void* qI, const void* w,
                            const void* kI, const int32_t* idx, int k_pad, const float* lse_cmp, const int32_t* cu,
                            const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H, int d, int H_I,
                            int d_I, int ratio, float scale, csa_dtype_t dtype, float* kl_sum, float* kl_per_query,
                            int32_t* n_valid, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return indexer_kl_common(h, q, kv_cmp, qI, w, kI, idx, k_pad, lse_cmp, cu, cu_cmp, B, T_cap, max_seqlen, H, d, H_I,
                           d_I, ratio, scale, dtype, kl_sum, kl_per_query, n_valid, ws, ws_bytes, nullptr, nullptr,
                           stream);
}

csa_status_t csa_indexer_kl_ex(csa_handle_t h, const void* q, const void* kv_cmp, const void* qI, const void* w,
                               const void* kI, const int32_t* idx, int k_pad, const float* lse_cmp, const int32_t* cu,
                               const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H, int d, int H_I,
                               int d_I, int ratio, float scale, csa_dtype_t dtype, float* kl_sum,
                               float* kl_per_query, int32_t* n_valid, void* ws, size_t ws_bytes,
                               float* teacher_lse, float* student_lse, cudaStream_t stream) {
  return indexer_kl_common(h, q, kv_cmp, qI, w, kI, idx, k_pad, lse_cmp, cu, cu_cmp, B, T_cap, max_seqlen, H, d, H_I,
                           d_I, ratio, scale, dtype, kl_sum, kl_per_query, n_valid, ws, ws_bytes, teacher_lse,
                           student_lse, stream);
}

csa_status_t csa_indexer_kl_bwd(csa_handle_t h, const void* q, const void* kv_cmp, const void* qI, const void* w,
                                const void* kI, const int32_t* idx, int k_pad, const float* lse_cmp,
                                const float* student_lse, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap, int max_seqlen, int H,
                                int d, int H_I, int d_I, int ratio, float scale, float grad_scale,
                                csa_dtype_t dtype, void* dqI, void* dw, float* dkI, cudaStream_t stream) {
  if (!h || !q || !kv_cmp || !qI || !w || !kI || !cu_cmp || !dqI || !dw || !dkI ||
      !packing_ok(cu, B, T_cap, max_seqlen))
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cmp) || !aligned16(qI) || !aligned16(kI) || !aligned16(dqI) ||
      !aligned16(dw) || !aligned16(dkI))
    return CSA_ERR_INVALID_ARG;
  if ((dtype != CSA_BF16 && dtype != CSA_FP32) || ratio < 1 || !(scale > 0.f) || !(grad_scale == grad_scale))
    return CSA_ERR_INVALID_ARG;
  if (idx != nullptr && k_pad < 1) return CSA_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || !pow2_in(H, 4, 128) || !pow2_in(H_I, 1, 8) || (d_I != 32 && d_I != 64))
    return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  csa::KLBwdArgs a{q, kv_cmp, qI, w, kI, idx, k_pad, lse_cmp, student_lse, cu, cu_cmp, B, T_cap, H, d, H_I, d_I, ratio,
                   h->cmp_rows > T_cap / ratio ? h->cmp_rows : T_cap / ratio, scale, grad_scale, dqI, dw, dkI,
                   h->status, h->pos0};
  return from_cuda(csa::launch_indexer_kl_bwd(a, dtype == CSA_FP32, stream));
}

csa_status_t csa_quantize_fp8(csa_handle_t h, const void* x, int64_t rows, int cols, csa_dtype_t dtype,
                              uint8_t* codes, float* scales, cudaStream_t stream) {
  if (!h || !x || !codes || !scales || rows < 0) return CSA_ERR_INVALID_ARG;
  if (dtype != CSA_BF16 && dtype != CSA_FP32) return CSA_ERR_INVALID_ARG;
  if (cols < 1 || cols > 256) return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  return from_cuda(csa::launch_quantize_fp8(x, rows, cols, dtype == CSA_FP32, codes, scales, stream));
}

csa_status_t csa_indexer_topk_fp8(csa_handle_t h, const uint8_t* qI, const float* qI_scale, const void* w,
                                  const uint8_t* kI, const float* kI_scale, const int32_t* cu, const int32_t* cu_cmp,
                                  int B, int T_cap, int max_seqlen, int H_I, int d_I, int ratio, int topk, int k_pad,
                                  csa_dtype_t dtype, int32_t* idx, cudaStream_t stream) {
  if (!h || !qI || !qI_scale || !w || !kI || !kI_scale || !cu_cmp || !idx || !packing_ok(cu, B, T_cap, max_seqlen))
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(qI) || !aligned16(kI) || !aligned16(idx)) return CSA_ERR_INVALID_ARG;
  if (ratio < 1 || topk < 1 || k_pad < topk) return CSA_ERR_INVALID_ARG;
  if (dtype != CSA_BF16 || H_I != 8 || d_I != 64 || k_pad > 8192) return CSA_ERR_UNSUPPORTED;
  const int max_vis = max_seqlen / ratio;
  if (!csa::indexer_topk_tc_supported(H_I, d_I, max_vis, false)) return CSA_ERR_UNSUPPORTED;
  DeviceGuard g(h->device);
  if (!g.ok) return CSA_ERR_CUDA;
  return from_cuda(csa::launch_indexer_topk_fp8_full(qI, qI_scale, w, kI, kI_scale, cu, cu_cmp, B, T_cap, max_vis,
                                                     ratio, topk, k_pad, idx, h->status, stream, h->pos0,
                                                     h->cmp_rows));
}

}  // extern "C"

namespace csa {
// Device of a handle (for entry points defined in other translation units).
int handle_device(csa_handle_t h) { return h->device; }
}  // namespace csa
