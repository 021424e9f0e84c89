// indexer_kl_bwd.cu -- backward of the indexer KL auxiliary loss.
//
// "DeepSeek-V4 Attention Training Systems": §3 (L_I = sum_t KL(p_t || q_t) over
// C_t), §8.2 ("indexer backward": the discrete top-k has no LM-loss gradient,
// so the indexer learns only through this loss; "teacher operands are
// detached"; the page runs it eagerly inside the forward with a unit loss
// gradient and applies the loss scale later), §9 (FP32 loss math).
//
// With the teacher p(j) = (1/H) sum_h softmax_{C_t}(scale q_h . K_j) and the
// student q(j) = softmax_{C_t}(i_j), i_j = sum_h w_h ReLU(a_hj), a_hj = qI_h . kI_j,
// the loss gradient of logit i_j is g_j = grad_scale (q(j) - p(j)), and
//   dw_h = sum_j g_j ReLU(a_hj),   dqI_h = w_h sum_j g_j [a_hj > 0] kI_j,
//   dkI_j += sum_h g_j w_h [a_hj > 0] qI_h          (float32, red.global.add).
// One CTA per query row, warps of 16 teacher heads as in the forward kernel.
// Pass 1 (the teacher's per-head log-sum-exp is skipped when the forward's
// lse_cmp is given) also takes the student's log-sum-exp over C_t; pass 2
// recomputes S = Q K^T on mma.sync for p(j) and the indexer dots for i_j, then
// forms g and the three gradient terms with the tile in shared memory.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sm80.cuh"
#include "tile_sm80.cuh"

namespace csa {

namespace {
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
}  // namespace

template <typename TIn, int D, int NW, int DI>
__global__ void __launch_bounds__(NW * 32)
indexer_kl_bwd_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k_cmp, const TIn* __restrict__ qI,
                      const TIn* __restrict__ w, const TIn* __restrict__ kI, const int32_t* __restrict__ idx,
                      int k_pad, const float* __restrict__ lse_cmp, const int32_t* __restrict__ cu,
                      const int32_t* __restrict__ cu_cmp, int B, int H, int H_I, int r, float scale_log2,
                      float grad_scale, TIn* __restrict__ dqI, TIn* __restrict__ dw, float* __restrict__ dkI,
                      int* status) {
  constexpr int kStride = AttnSmem<D>::kStride;
  constexpr int kRows = NW * 16;
  constexpr int kThreads = NW * 32;
  constexpr int kHK = 8 * kKeys;                         // (indexer head, key) pairs of a tile
  constexpr int kIterHK = kHK / kThreads;
  constexpr int kIterDQ = (8 * DI + kThreads - 1) / kThreads;
  constexpr int kChunks = kKeys * (DI / 8);              // (key, 8-channel chunk) pairs of a tile
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sK = sQ + kRows * kStride;                       // [2][kKeys][kStride]
  __nv_bfloat16* sKI = sK + 2 * kKeys * kStride;                  // [2][kKeys][DI]
  float* sQI = reinterpret_cast<float*>(sKI + 2 * kKeys * DI);    // [8][DI]
  float* sW = sQI + 8 * DI;                                       // [8]
  float* sPsum = sW + 8;                                          // [NW][kKeys]
  float* sA = sPsum + NW * kKeys;                                 // [8][kKeys] ReLU(a_hj)
  float* sG = sA + kHK;                                           // [kKeys] g_j
  float* sRed = sG + kKeys;                                       // [max(kHK, 2 kThreads)]
  __shared__ int s_rows[2][kKeys];
  __shared__ float s_lse_i;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int b = owner_sequence(cu, B, row);
  auto write_zero = [&]() {
    for (int i = tid; i < H_I * DI; i += kThreads) dqI[(int64_t)row * H_I * DI + i] = from_f32<TIn>(0.f);
    for (int i = tid; i < H_I; i += kThreads) dw[(int64_t)row * H_I + i] = from_f32<TIn>(0.f);
  };
  if (b < 0) { write_zero(); return; }
  const int t = row - __ldg(cu + b);
  const int nvis = r > 0 ? (t + 1) / r : 0;
  const int cmp0 = __ldg(cu_cmp + b);
  const bool dense = idx == nullptr;
  const int n_slots = dense ? nvis : k_pad;
  const int ntiles = (n_slots + kKeys - 1) / kKeys;

  for (int i = tid; i < kRows * (D / 8); i += kThreads) {
    const int h = i / (D / 8), c = i - h * (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h < H) v = Load8<TIn>::run(q + ((int64_t)row * H + h) * D + c * 8);
    *reinterpret_cast<uint4*>(sQ + h * kStride + c * 8) = v;
  }
  for (int i = tid; i < 8 * DI; i += kThreads) {
    const int h = i / DI, c = i - h * DI;
    sQI[i] = h < H_I ? to_f32(qI[((int64_t)row * H_I + h) * DI + c]) : 0.f;
  }
  if (tid < 8) sW[tid] = tid < H_I ? to_f32(w[(int64_t)row * H_I + tid]) : 0.f;

  const int cmp_limit = __ldg(cu_cmp + B);
  auto resolve = [&](int it, int buf) {
    for (int kk = tid; kk < kKeys; kk += kThreads) {
      int rr = -1;
      const int slot = it * kKeys + kk;
      if (dense) {
        if (slot < nvis) rr = cmp0 + slot;
      } else if (slot < k_pad) {
        const int g = __ldg(idx + (int64_t)row * k_pad + slot);
        if (g >= 0) {
          if (g < cmp0 || g >= cmp0 + nvis) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
          else rr = g;
        }
      }
      s_rows[buf][kk] = rr;
    }
  };
  auto issue = [&](int buf) {
    gather_tile<TIn, D>(k_cmp, k_cmp, false, s_rows[buf], cmp_limit, sK + buf * kKeys * kStride, nullptr, tid,
                        kThreads);
    for (int i = tid; i < kKeys * (DI / 8); i += kThreads) {
      const int k = i / (DI / 8), c = i - k * (DI / 8);
      const int rr = s_rows[buf][k] < cmp_limit ? s_rows[buf][k] : -1;
      __nv_bfloat16* dst = sKI + (buf * kKeys + k) * DI + c * 8;
      if constexpr (sizeof(TIn) == 2) {
        cp_async_16_zfill(smem_u32(dst), kI + (int64_t)(rr < 0 ? 0 : rr) * DI + c * 8, rr >= 0);
      } else {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rr >= 0) v = Load8<TIn>::run(kI + (int64_t)rr * DI + c * 8);
        *reinterpret_cast<uint4*>(dst) = v;
      }
    }
  };
  // ReLU(a_hj) of the tile's (head, key) pairs into sA
  auto indexer_dots = [&](int buf) {
    const __nv_bfloat16* tKI = sKI + buf * kKeys * DI;
    for (int wi = tid; wi < kHK; wi += kThreads) {
      const int k = wi & (kKeys - 1), h = wi / kKeys;
      float dot = 0.f;
      if (h < H_I) {
#pragma unroll 8
        for (int c = 0; c < DI; ++c) dot = fmaf(sQI[h * DI + c], __bfloat162float(tKI[k * DI + c]), dot);
      }
      sA[wi] = fmaxf(dot, 0.f);
    }
  };

  // ---- pass 1: per-head teacher log-sum-exp and the student's over C_t ----
  float lse2[2] = {-INFINITY, -INFINITY};
  const bool have_lse = (!dense) && lse_cmp != nullptr;
  if (have_lse) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int h = warp * 16 + (lane >> 2) + i * 8;
      lse2[i] = h < H ? __ldg(lse_cmp + (int64_t)row * H + h) * kLog2e : -INFINITY;
    }
  }
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float mi = -INFINITY, li = 0.f;  // student log-sum-exp (natural units), per key thread
  if (ntiles > 0) { resolve(0, 0); __syncthreads(); issue(0); }
  cp_async_commit();
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntiles) { resolve(it + 1, buf ^ 1); __syncthreads(); issue(buf ^ 1); }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (!have_lse) {
      float s[8][4];
      qk_tile<D>(sQ, sK + buf * kKeys * kStride, warp, lane, s);
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = n * 8 + (lane & 3) * 2 + (e & 1);
          const float v = s_rows[buf][key] >= 0 ? s[n][e] * scale_log2 : -INFINITY;
          s[n][e] = v;
          tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
        }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 1));
        tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 2));
        const float mnew = fmaxf(m_run[i], tmax[i]);
        const float muse = mnew == -INFINITY ? 0.f : mnew;
        l_run[i] *= exp2f(m_run[i] - muse);
        m_run[i] = mnew;
#pragma unroll
        for (int n = 0; n < 8; ++n) l_run[i] += exp2f(s[n][2 * i] - muse) + exp2f(s[n][2 * i + 1] - muse);
      }
    }
    indexer_dots(buf);
    __syncthreads();
    for (int kk = tid; kk < kKeys; kk += kThreads) {
      if (s_rows[buf][kk] < 0) continue;
      float il = 0.f;
#pragma unroll
      for (int h = 0; h < 8; ++h) il = fmaf(sW[h], sA[h * kKeys + kk], il);
      if (il > mi) { li = li * __expf(mi - il) + 1.f; mi = il; }
      else li += __expf(il - mi);
    }
    __syncthreads();
  }
  if (!have_lse) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float l = l_run[i];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const int h = warp * 16 + (lane >> 2) + i * 8;
      lse2[i] = (l > 0.f && h < H) ? m_run[i] + __log2f(l) : -INFINITY;  // padding heads add nothing
    }
  }
  sRed[tid] = mi;
  sRed[kThreads + tid] = li;
  __syncthreads();
  if (tid == 0) {
    float M = -INFINITY;
    for (int k = 0; k < kThreads; ++k) M = fmaxf(M, sRed[k]);
    float Ls = 0.f;
    for (int k = 0; k < kThreads; ++k)
      if (sRed[k] != -INFINITY) Ls += sRed[kThreads + k] * __expf(sRed[k] - M);
    s_lse_i = Ls > 0.f ? M + __logf(Ls) : -INFINITY;
  }
  __syncthreads();
  const float lse_i = s_lse_i;
  if (lse_i == -INFINITY) { write_zero(); return; }   // empty C_t: no loss, no gradient (uniform exit)

  // ---- pass 2: g_j = grad_scale (q(j) - p(j)) and the gradient terms ----
  const float inv_h = 1.f / (float)H;
  float dwp[kIterHK];
  float dqp[kIterDQ];
#pragma unroll
  for (int m = 0; m < kIterHK; ++m) dwp[m] = 0.f;
#pragma unroll
  for (int m = 0; m < kIterDQ; ++m) dqp[m] = 0.f;
  if (ntiles > 0) { resolve(0, 0); __syncthreads(); issue(0); }
  cp_async_commit();
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntiles) { resolve(it + 1, buf ^ 1); __syncthreads(); issue(buf ^ 1); }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    float s[8][4];
    qk_tile<D>(sQ, sK + buf * kKeys * kStride, warp, lane, s);
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = 0.f;
        if (lse2[0] != -INFINITY) v += exp2f(s[n][e] * scale_log2 - lse2[0]);
        if (lse2[1] != -INFINITY) v += exp2f(s[n][2 + e] * scale_log2 - lse2[1]);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (lane < 4) sPsum[warp * kKeys + n * 8 + lane * 2 + e] = v;
      }
    }
    indexer_dots(buf);
    __syncthreads();
    for (int kk = tid; kk < kKeys; kk += kThreads) {
      float g = 0.f;
      if (s_rows[buf][kk] >= 0) {
        float p = 0.f;
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) p += sPsum[ww * kKeys + kk];
        float il = 0.f;
#pragma unroll
        for (int h = 0; h < 8; ++h) il = fmaf(sW[h], sA[h * kKeys + kk], il);
        g = grad_scale * (__expf(il - lse_i) - p * inv_h);
      }
      sG[kk] = g;
    }
    __syncthreads();
    // dw_h += g_j ReLU(a_hj): thread-owned (head, key) pairs, summed over keys at the end
#pragma unroll
    for (int m = 0; m < kIterHK; ++m) {
      const int wi = tid + m * kThreads;
      dwp[m] = fmaf(sG[wi & (kKeys - 1)], sA[wi], dwp[m]);
    }
    // dqI_h[c] += sum_j g_j w_h [a_hj > 0] kI_j[c]
    const __nv_bfloat16* tKI = sKI + buf * kKeys * DI;
#pragma unroll
    for (int m = 0; m < kIterDQ; ++m) {
      const int o = tid + m * kThreads;
      if (o < 8 * DI) {
        const int h = o / DI, c = o - h * DI;
        float acc = 0.f;
        for (int k = 0; k < kKeys; ++k)
          if (sA[h * kKeys + k] > 0.f) acc = fmaf(sG[k], __bfloat162float(tKI[k * DI + c]), acc);
        dqp[m] = fmaf(sW[h], acc, dqp[m]);
      }
    }
    // dkI_j[c0..c0+8) += sum_h g_j w_h [a_hj > 0] qI_h[c0..c0+8)
    for (int o = tid; o < kChunks; o += kThreads) {
      const int k = o / (DI / 8), c0 = (o - k * (DI / 8)) * 8;
      const int rr = s_rows[buf][k];
      const float g = sG[k];
      if (rr < 0 || g == 0.f) continue;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (!(sA[h * kKeys + k] > 0.f)) continue;
        const float cf = g * sW[h];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(cf, sQI[h * DI + c0 + e], acc[e]);
      }
      float* dst = dkI + (int64_t)rr * DI + c0;
      red_add_v4(dst, acc[0], acc[1], acc[2], acc[3]);
      red_add_v4(dst + 4, acc[4], acc[5], acc[6], acc[7]);
    }
    __syncthreads();
  }
  // dw: the (head, key) partials summed over keys in a fixed order
#pragma unroll
  for (int m = 0; m < kIterHK; ++m) sA[tid + m * kThreads] = dwp[m];
  __syncthreads();
  for (int h = tid; h < H_I; h += kThreads) {
    float sacc = 0.f;
    for (int k = 0; k < kKeys; ++k) sacc += sA[h * kKeys + k];
    dw[(int64_t)row * H_I + h] = from_f32<TIn>(sacc);
  }
#pragma unroll
  for (int m = 0; m < kIterDQ; ++m) {
    const int o = tid + m * kThreads;
    if (o < 8 * DI && o / DI < H_I) dqI[(int64_t)row * H_I * DI + o] = from_f32<TIn>(dqp[m]);
  }
}

template <typename TIn, int D, int NW, int DI>
static cudaError_t launch_kl_bwd_t(const KLBwdArgs& a, cudaStream_t stream) {
  constexpr int kStride = AttnSmem<D>::kStride;
  constexpr int kThreads = NW * 32;
  constexpr int kHK = 8 * kKeys;
  const size_t smem = (size_t)(NW * 16 + 2 * kKeys) * kStride * 2 + (size_t)2 * kKeys * DI * 2 +
                      ((size_t)8 * DI + 8 + NW * kKeys + kHK + kKeys + (kHK > 2 * kThreads ? kHK : 2 * kThreads)) * 4;
  auto kern = indexer_kl_bwd_kernel<TIn, D, NW, DI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  constexpr float kLog2e = 1.4426950408889634f;
  kern<<<a.T_cap, kThreads, smem, stream>>>(
      static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k_cmp), static_cast<const TIn*>(a.qI),
      static_cast<const TIn*>(a.w), static_cast<const TIn*>(a.kI), a.idx, a.k_pad, a.lse_cmp, a.cu, a.cu_cmp, a.B,
      a.H, a.H_I, a.r, a.scale * kLog2e, a.grad_scale, static_cast<TIn*>(a.dqI), static_cast<TIn*>(a.dw), a.dkI,
      a.status);
  return cudaGetLastError();
}

template <typename TIn, int D, int DI>
static cudaError_t kl_bwd_heads(const KLBwdArgs& a, cudaStream_t stream) {
  switch ((a.H + 15) / 16) {
    case 1: return launch_kl_bwd_t<TIn, D, 1, DI>(a, stream);
    case 2: return launch_kl_bwd_t<TIn, D, 2, DI>(a, stream);
    case 4: return launch_kl_bwd_t<TIn, D, 4, DI>(a, stream);
    case 8: return launch_kl_bwd_t<TIn, D, 8, DI>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename TIn>
static cudaError_t kl_bwd_dims(const KLBwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.d_I == 32 ? kl_bwd_heads<TIn, 64, 32>(a, stream) : kl_bwd_heads<TIn, 64, 64>(a, stream);
  return a.d_I == 32 ? kl_bwd_heads<TIn, 128, 32>(a, stream) : kl_bwd_heads<TIn, 128, 64>(a, stream);
}

cudaError_t launch_indexer_kl_bwd(const KLBwdArgs& a, bool fp32, cudaStream_t stream) {
  if (a.T_cap <= 0) return cudaSuccess;
  cudaError_t err = cudaMemsetAsync(a.dkI, 0, (size_t)a.n_cmp_cap * a.d_I * 4, stream);
  if (err != cudaSuccess) return err;
  return fp32 ? kl_bwd_dims<float>(a, stream) : kl_bwd_dims<__nv_bfloat16>(a, stream);
}

}  // namespace csa
