// indexer_kl.cu -- the indexer KL auxiliary loss.
//
// "DeepSeek-V4 Attention Training Systems": §3 (L_I = sum_t KL(Softmax(a_{t,C_t})
// || Softmax(i_{t,C_t})), C_t the full visible history in the dense-loss phase
// or the selected set in sparse-loss mode), §2 phase table (the dense teacher
// of the sparse warm-up is ~O(L^2/4) score work), §8.2 ("recompute sparse/dense
// teacher scores for the indexer loss"), §9 (FP32 loss math).
//
// Teacher: p(j) = (1/H) sum_h softmax_{C_t}(scale q_h . K_j); student: softmax of
// the indexer logits over C_t.  Per query row one CTA; warps split the heads as
// in the attention kernel.  Pass 1 runs the per-head online log-sum-exp; pass 2 recomputes the
// scores, forms p(j) by summing exp2(s - lse) over heads (shuffles within a
// warp, shared memory across warps), computes the indexer logit of each key
// and accumulates sum p log p, sum p i and the student's log-sum-exp, so that
// KL_t = sum p log p - sum p i + lse_i.  A second kernel adds the per-query
// values in a fixed order (deterministic).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sm80.cuh"
#include "tile_sm80.cuh"

namespace csa {

template <typename TIn, int D, int NW, int DI>
__global__ void __launch_bounds__(NW * 32)
indexer_kl_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k_cmp, const TIn* __restrict__ qI,
                  const TIn* __restrict__ w, const TIn* __restrict__ kI, const int32_t* __restrict__ idx,
                  int k_pad, const float* __restrict__ lse_cmp, const int32_t* __restrict__ cu,
                  const int32_t* __restrict__ cu_cmp, int B, int H, int H_I, int r, float scale_log2,
                  float* __restrict__ kl_rows, int32_t* __restrict__ csize, int* status,
                  float* __restrict__ teacher_lse, float* __restrict__ student_lse,
                  const int32_t* __restrict__ pos0) {
  constexpr int kStride = AttnSmem<D>::kStride;
  constexpr int kRows = NW * 16;
  constexpr int kThreads = NW * 32;
  constexpr float kLn2 = 0.6931471805599453f;
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sK = sQ + kRows * kStride;                       // [2][kKeys][kStride]
  __nv_bfloat16* sKI = sK + 2 * kKeys * kStride;                  // [2][kKeys][DI]
  float* sQI = reinterpret_cast<float*>(sKI + 2 * kKeys * DI);    // [8][DI]
  float* sW = sQI + 8 * DI;                                       // [8]
  float* sPsum = sW + 8;                                          // [NW][kKeys]
  float* sIlog = sPsum + NW * kKeys;                              // [kKeys]
  float* sRed = sIlog + kKeys;                                    // [kThreads * 4]
  __shared__ int s_rows[2][kKeys];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int b = owner_sequence(cu, B, row);
  if (b < 0) {
    if (tid == 0) {
      kl_rows[row] = 0.f;
      csize[row] = 0;
      if (student_lse) student_lse[row] = -INFINITY;
    }
    if (teacher_lse)
      for (int h = tid; h < H; h += kThreads) teacher_lse[(int64_t)row * H + h] = -INFINITY;
    return;
  }
  const int t = row - __ldg(cu + b);
  const int p0 = pos0 ? __ldg(pos0 + b) : 0;  // position of the sequence's first row here
  const int nvis = r > 0 ? (t + p0 + 1) / r : 0;
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

  int count = 0;  // |C_t| entries resolved by this thread (summed at the end)
  const int cmp_limit = __ldg(cu_cmp + B);
  auto resolve = [&](int it, int buf, bool tally) {
    for (int kk = tid; kk < kKeys; kk += kThreads) {
      int rr = -1;
      const int slot = it * kKeys + kk;
      if (dense) {
        if (slot < nvis) rr = cmp0 + slot;
      } else if (slot < k_pad) {
        const int g = __ldg(idx + (int64_t)row * k_pad + slot);
        if (g >= 0) {
          if (g < cmp0 || g >= cmp0 + nvis) { if (tally) raise_status(status, CSA_ERR_DEVICE_BOUNDS); }
          else rr = g;
        }
      }
      s_rows[buf][kk] = rr;
      if (tally && rr >= 0) ++count;
    }
  };
  auto issue = [&](int buf, bool with_ki) {
    gather_tile<TIn, D>(k_cmp, k_cmp, false, s_rows[buf], cmp_limit, sK + buf * kKeys * kStride, nullptr, tid,
                        kThreads);
    if (with_ki) {
      // indexer key rows: DI bf16 = DI/8 chunks per row
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
    }
  };

  // per-head log2 normaliser over C_t for the two rows this thread holds (the
  // exact one: a given lse_cmp only serves the tensor-core kernel as a reference)
  float lse2[2] = {-INFINITY, -INFINITY};
  (void)lse_cmp;
  {
    // ---- pass 1: per-head online log-sum-exp over C_t ----
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    if (ntiles > 0) { resolve(0, 0, false); __syncthreads(); issue(0, false); }
    cp_async_commit();
    for (int it = 0; it < ntiles; ++it) {
      const int buf = it & 1;
      if (it + 1 < ntiles) { resolve(it + 1, buf ^ 1, false); __syncthreads(); issue(buf ^ 1, false); }
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
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
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float l = l_run[i];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const int h = warp * 16 + (lane >> 2) + i * 8;
      lse2[i] = (l > 0.f && h < H) ? m_run[i] + __log2f(l) : -INFINITY;  // padding heads add nothing
    }
  }
  if (teacher_lse != nullptr && (lane & 3) == 0) {  // natural units, for the indexer backward
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int h = warp * 16 + (lane >> 2) + i * 8;
      if (h < H) teacher_lse[(int64_t)row * H + h] = lse2[i] * kLn2;
    }
  }

  // ---- pass 2: teacher p(j), student logits, KL accumulators ----
  float accA = 0.f, accB = 0.f;            // sum p ln p, sum p i    (threads < kKeys)
  float mi = -INFINITY, li = 0.f;          // student log-sum-exp (natural units)
  const float inv_h = 1.f / (float)H;
  if (ntiles > 0) { resolve(0, 0, true); __syncthreads(); issue(0, true); }
  cp_async_commit();
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntiles) { resolve(it + 1, buf ^ 1, true); __syncthreads(); issue(buf ^ 1, true); }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    float s[8][4];
    qk_tile<D>(sQ, sK + buf * kKeys * kStride, warp, lane, s);
    // column sums of exp2(s - lse2) over this warp's heads
    float cs[8][2];
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
        cs[n][e] = v;
      }
    }
    if (lane < 4) {
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        sPsum[warp * kKeys + n * 8 + lane * 2] = cs[n][0];
        sPsum[warp * kKeys + n * 8 + lane * 2 + 1] = cs[n][1];
      }
    }
    // indexer logits of the tile's keys: thread (key, head group)
    {
      const __nv_bfloat16* tKI = sKI + buf * kKeys * DI;
      for (int wi = tid; wi < kKeys * 8; wi += kThreads) {
        const int k = wi & (kKeys - 1), h = wi / kKeys;
        float v = 0.f;
        if (h < H_I) {
          float dot = 0.f;
#pragma unroll 8
          for (int c = 0; c < DI; ++c) dot = fmaf(sQI[h * DI + c], __bfloat162float(tKI[k * DI + c]), dot);
          v = sW[h] * fmaxf(dot, 0.f);
        }
        sRed[wi] = v;
      }
    }
    __syncthreads();
    for (int kk = tid; kk < kKeys; kk += kThreads) {
      if (s_rows[buf][kk] < 0) continue;
      float p = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) p += sPsum[ww * kKeys + kk];
      p *= inv_h;
      float il = 0.f;
      for (int h = 0; h < 8; ++h) il += sRed[h * kKeys + kk];
      if (p > 0.f) accA += p * __logf(p);
      accB = fmaf(p, il, accB);
      if (il > mi) { li = li * __expf(mi - il) + 1.f; mi = il; }
      else li += __expf(il - mi);
    }
    __syncthreads();
  }
  // block reduction of the per-thread partials (kThreads <= 256 entries each)
  sRed[tid] = accA;
  sRed[kThreads + tid] = accB;
  sRed[2 * kThreads + tid] = mi;
  sRed[3 * kThreads + tid] = li;
  reinterpret_cast<int*>(sPsum)[tid] = count;
  __syncthreads();
  if (tid == 0) {
    float A = 0.f, Bs = 0.f, M = -INFINITY;
    int n = 0;
    for (int k = 0; k < kThreads; ++k) {
      A += sRed[k];
      Bs += sRed[kThreads + k];
      M = fmaxf(M, sRed[2 * kThreads + k]);
      n += reinterpret_cast<int*>(sPsum)[k];
    }
    float Ls = 0.f;
    for (int k = 0; k < kThreads; ++k)
      if (sRed[2 * kThreads + k] != -INFINITY) Ls += sRed[3 * kThreads + k] * __expf(sRed[2 * kThreads + k] - M);
    const float kl = n > 0 ? A - Bs + (M + __logf(Ls)) : 0.f;
    kl_rows[row] = kl;
    csize[row] = n;
    if (student_lse) student_lse[row] = n > 0 ? M + __logf(Ls) : -INFINITY;
  }
  (void)kLn2;
}

// kl_sum = sum of kl_rows in a fixed order (double accumulation); n_valid.
__global__ void __launch_bounds__(1024)
kl_finalize_kernel(const float* __restrict__ kl_rows, const int32_t* __restrict__ csize, int T_cap,
                   float* kl_sum, int32_t* n_valid) {
  __shared__ double s_sum[1024];
  __shared__ int s_cnt[1024];
  double acc = 0.0;
  int cnt = 0;
  for (int i = threadIdx.x; i < T_cap; i += blockDim.x) {
    acc += (double)kl_rows[i];
    cnt += csize[i] > 0;
  }
  s_sum[threadIdx.x] = acc;
  s_cnt[threadIdx.x] = cnt;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) {
      s_sum[threadIdx.x] += s_sum[threadIdx.x + o];
      s_cnt[threadIdx.x] += s_cnt[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *kl_sum = (float)s_sum[0];
    if (n_valid) *n_valid = s_cnt[0];
  }
}

template <typename TIn, int D, int NW, int DI>
static cudaError_t launch_kl_t(const KLArgs& a, cudaStream_t stream) {
  constexpr int kStride = AttnSmem<D>::kStride;
  const size_t smem = (size_t)(NW * 16 + 2 * kKeys) * kStride * 2 + (size_t)2 * kKeys * DI * 2 +
                      sizeof(float) * (8 * DI + 8 + NW * kKeys + kKeys + NW * 32 * 4 + 8 * kKeys);
  auto kern = indexer_kl_kernel<TIn, D, NW, DI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  constexpr float kLog2e = 1.4426950408889634f;
  if (a.T_cap > 0) {
    kern<<<a.T_cap, NW * 32, smem, stream>>>(
        static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k_cmp), static_cast<const TIn*>(a.qI),
        static_cast<const TIn*>(a.w), static_cast<const TIn*>(a.kI), a.idx, a.k_pad, a.lse_cmp, a.cu,
        a.cu_cmp, a.B, a.H, a.H_I, a.r, a.scale * kLog2e, a.kl_rows, a.csize, a.status, a.teacher_lse,
        a.student_lse, a.pos0);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  kl_finalize_kernel<<<1, 1024, 0, stream>>>(a.kl_rows, a.csize, a.T_cap, a.kl_sum, a.n_valid);
  return cudaGetLastError();
}

template <typename TIn, int D, int DI>
static cudaError_t kl_heads(const KLArgs& a, cudaStream_t stream) {
  switch ((a.H + 15) / 16) {
    case 1: return launch_kl_t<TIn, D, 1, DI>(a, stream);
    case 2: return launch_kl_t<TIn, D, 2, DI>(a, stream);
    case 4: return launch_kl_t<TIn, D, 4, DI>(a, stream);
    case 8: return launch_kl_t<TIn, D, 8, DI>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename TIn, int D>
static cudaError_t kl_di(const KLArgs& a, cudaStream_t stream) {
  return a.d_I == 32 ? kl_heads<TIn, D, 32>(a, stream) : kl_heads<TIn, D, 64>(a, stream);
}

cudaError_t launch_indexer_kl(const KLArgs& a, bool fp32, cudaStream_t stream) {
  // the dense teacher at 64 x 128 heads / 8 x 64 indexer (bf16) runs on tcgen05 with TMA-fed tiles
  if (indexer_kl_dense_tc_supported(a, fp32)) {
    cudaError_t err = launch_indexer_kl_dense_tc(a, stream);
    if (err != cudaSuccess) return err;
    kl_finalize_kernel<<<1, 1024, 0, stream>>>(a.kl_rows, a.csize, a.T_cap, a.kl_sum, a.n_valid);
    return cudaGetLastError();
  }
  // the selected-set teacher at the same shapes, with a reference normaliser from the attention
  if (indexer_kl_sparse_tc_supported(a, fp32)) {
    cudaError_t err = launch_indexer_kl_sparse_tc(a, stream);
    if (err != cudaSuccess) return err;
    kl_finalize_kernel<<<1, 1024, 0, stream>>>(a.kl_rows, a.csize, a.T_cap, a.kl_sum, a.n_valid);
    return cudaGetLastError();
  }
  if (fp32) return a.d == 64 ? kl_di<float, 64>(a, stream) : kl_di<float, 128>(a, stream);
  return a.d == 64 ? kl_di<__nv_bfloat16, 64>(a, stream) : kl_di<__nv_bfloat16, 128>(a, stream);
}

}  // namespace csa
