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
// forms g.  The indexer dots a = qI kI^T, dqI += C kI and the key-block
// gradient dkI = C^T qI (C[h, j] = g_j w_h [a_hj > 0] as a bf16 tile, the 8
// indexer heads padded to 16 rows) are mma.sync products too.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sm80.cuh"
#include "tile_sm80.cuh"

namespace csa {

namespace {
__device__ __forceinline__ void red_add_v2(float* p, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};\n" ::"l"(p), "f"(a), "f"(b) : "memory");
}
}  // namespace

template <typename TIn, int D, int NW, int DI>
__global__ void __launch_bounds__(NW * 32)
indexer_kl_bwd_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k_cmp, const TIn* __restrict__ qI,
                      const TIn* __restrict__ w, const TIn* __restrict__ kI, const int32_t* __restrict__ idx,
                      int k_pad, const float* __restrict__ lse_cmp, const float* __restrict__ student_lse,
                      const int32_t* __restrict__ cu,
                      const int32_t* __restrict__ cu_cmp, int B, int H, int H_I, int r, float scale_log2,
                      float grad_scale, TIn* __restrict__ dqI, TIn* __restrict__ dw, float* __restrict__ dkI,
                      int* status,
                      const int32_t* __restrict__ pos0) {
  constexpr int kStride = AttnSmem<D>::kStride;
  constexpr int kRows = NW * 16;
  constexpr int kThreads = NW * 32;
  constexpr int kHK = 8 * kKeys;                         // (indexer head, key) pairs of a tile
  constexpr int kIterHK = kHK / kThreads;
  constexpr int kKIS = DI + 8;                           // bf16 row stride of the indexer rows (16 B pad)
  constexpr int kCS = kKeys + 8;                         // bf16 row stride of the coefficient tile
  constexpr int kDQB = DI / 16;                          // 16-channel blocks of dqI
  constexpr int kDQPerWarp = (kDQB + NW - 1) / NW;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sK = sQ + kRows * kStride;                       // [2][kKeys][kStride]
  __nv_bfloat16* sKI = sK + 2 * kKeys * kStride;                  // [2][kKeys][kKIS]
  __nv_bfloat16* sQIb = sKI + 2 * kKeys * kKIS;                   // [16][kKIS] (rows >= H_I zero)
  __nv_bfloat16* sC = sQIb + 16 * kKIS;                           // [16][kCS]  (rows >= 8 zero)
  float* sQI = reinterpret_cast<float*>(sC + 16 * kCS);           // [8][DI]
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
  for (int i = tid; i < 16 * DI; i += kThreads) {
    const int h = i / DI, c = i - h * DI;
    const float v = h < H_I ? to_f32(qI[((int64_t)row * H_I + h) * DI + c]) : 0.f;
    if (h < 8) sQI[i] = v;
    sQIb[h * kKIS + c] = __float2bfloat16_rn(v);
  }
  for (int i = tid; i < 16 * kCS; i += kThreads) sC[i] = __float2bfloat16_rn(0.f);
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
      __nv_bfloat16* dst = sKI + (buf * kKeys + k) * kKIS + c * 8;
      if constexpr (sizeof(TIn) == 2) {
        cp_async_16_zfill(smem_u32(dst), kI + (int64_t)(rr < 0 ? 0 : rr) * DI + c * 8, rr >= 0);
      } else {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rr >= 0) v = Load8<TIn>::run(kI + (int64_t)rr * DI + c * 8);
        *reinterpret_cast<uint4*>(dst) = v;
      }
    }
  };
  // ReLU(a_hj) of the tile's (head, key) pairs into sA: a = qI kI^T on mma.sync
  // (indexer heads on M, padded to 16; 16 keys per warp and step)
  auto indexer_dots = [&](int buf) {
    const __nv_bfloat16* tKI = sKI + buf * kKeys * kKIS;
    for (int np = warp; np < kKeys / 16; np += NW) {
      float c2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < DI / 16; ++kk) {
        uint32_t a[4], bq[4];
        ldmatrix_x4(smem_u32(sQIb + (lane & 15) * kKIS + kk * 16 + (lane >> 4) * 8), a[0], a[1], a[2], a[3]);
        const int key = np * 16 + (lane & 7) + (lane >> 4) * 8;
        const int col = kk * 16 + ((lane >> 3) & 1) * 8;
        ldmatrix_x4(smem_u32(tKI + key * kKIS + col), bq[0], bq[1], bq[2], bq[3]);
        mma_bf16_16816(c2[0], a, bq);
        mma_bf16_16816(c2[1], a, bq + 2);
      }
      const int h = lane >> 2;   // rows 0..7 hold the 8 indexer heads
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = np * 16 + j * 8 + (lane & 3) * 2;
        sA[h * kKeys + key] = fmaxf(c2[j][0], 0.f);
        sA[h * kKeys + key + 1] = fmaxf(c2[j][1], 0.f);
      }
    }
  };

  // ---- pass 1: per-head teacher log-sum-exp and the student's over C_t (skipped when
  // the forward handed both over) ----
  float lse2[2] = {-INFINITY, -INFINITY};
  const bool have_lse = lse_cmp != nullptr;
  const bool one_pass = have_lse && student_lse != nullptr;
  if (have_lse) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int h = warp * 16 + (lane >> 2) + i * 8;
      lse2[i] = h < H ? __ldg(lse_cmp + (int64_t)row * H + h) * kLog2e : -INFINITY;
    }
  }
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float mi = -INFINITY, li = 0.f;  // student log-sum-exp (natural units), per key thread
  const int ntiles1 = one_pass ? 0 : ntiles;
  if (ntiles1 > 0) { resolve(0, 0); __syncthreads(); issue(0); }
  cp_async_commit();
  for (int it = 0; it < ntiles1; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntiles1) { resolve(it + 1, buf ^ 1); __syncthreads(); issue(buf ^ 1); }
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
    s_lse_i = one_pass ? __ldg(student_lse + row) : (Ls > 0.f ? M + __logf(Ls) : -INFINITY);
  }
  __syncthreads();
  const float lse_i = s_lse_i;
  if (lse_i == -INFINITY) { write_zero(); return; }   // empty C_t: no loss, no gradient (uniform exit)

  // ---- pass 2: g_j = grad_scale (q(j) - p(j)) and the gradient terms ----
  const float inv_h = 1.f / (float)H;
  float dwp[kIterHK];
  float dqf[kDQPerWarp][2][4];   // dqI fragments of this warp's 16-channel blocks (rows = heads)
#pragma unroll
  for (int m = 0; m < kIterHK; ++m) dwp[m] = 0.f;
#pragma unroll
  for (int i = 0; i < kDQPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) dqf[i][j][0] = dqf[i][j][1] = dqf[i][j][2] = dqf[i][j][3] = 0.f;
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
    // coefficient tile C[h][j] = g_j w_h [a_hj > 0] (bf16, rows 0..7)
    for (int wi = tid; wi < kHK; wi += kThreads) {
      const int k = wi & (kKeys - 1), h = wi / kKeys;
      sC[h * kCS + k] = __float2bfloat16_rn(sA[wi] > 0.f ? sG[k] * sW[h] : 0.f);
    }
    __syncthreads();
    const __nv_bfloat16* tKI = sKI + buf * kKeys * kKIS;
    // dqI += C kI: M = heads (16), N = 16 channels per block, K = the tile's keys
#pragma unroll
    for (int i = 0; i < kDQPerWarp; ++i) {
      const int blk = warp + i * NW;
      if (blk < kDQB) {
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          uint32_t a[4], bk[4];
          ldmatrix_x4(smem_u32(sC + (lane & 15) * kCS + kk * 16 + (lane >> 4) * 8), a[0], a[1], a[2], a[3]);
          const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int col = blk * 16 + (lane >> 4) * 8;
          ldmatrix_x4_trans(smem_u32(tKI + key * kKIS + col), bk[0], bk[1], bk[2], bk[3]);
          mma_bf16_16816(dqf[i][0], a, bk);
          mma_bf16_16816(dqf[i][1], a, bk + 2);
        }
      }
    }
    // dkI = C^T qI for 16-key blocks: M = keys, N = channels, K = heads (16)
    for (int kg = warp; kg < kKeys / 16; kg += NW) {
      const int m0 = kg * 16;
      uint32_t a[4];
      const int mi = lane >> 3;
      ldmatrix_x4_trans(smem_u32(sC + ((mi >> 1) * 8 + (lane & 7)) * kCS + m0 + (mi & 1) * 8), a[0], a[1], a[2],
                        a[3]);
      float acc[DI / 8][4];
#pragma unroll
      for (int nd = 0; nd < DI / 16; ++nd) {
        uint32_t bq[4];
        const int hr = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int col = nd * 16 + (lane >> 4) * 8;
        ldmatrix_x4_trans(smem_u32(sQIb + hr * kKIS + col), bq[0], bq[1], bq[2], bq[3]);
        acc[2 * nd][0] = acc[2 * nd][1] = acc[2 * nd][2] = acc[2 * nd][3] = 0.f;
        acc[2 * nd + 1][0] = acc[2 * nd + 1][1] = acc[2 * nd + 1][2] = acc[2 * nd + 1][3] = 0.f;
        mma_bf16_16816(acc[2 * nd], a, bq);
        mma_bf16_16816(acc[2 * nd + 1], a, bq + 2);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = m0 + (lane >> 2) + i * 8;
        const int rr = s_rows[buf][k];
        if (rr < 0 || sG[k] == 0.f) continue;
#pragma unroll
        for (int nd8 = 0; nd8 < DI / 8; ++nd8)
          red_add_v2(dkI + (int64_t)rr * DI + nd8 * 8 + (lane & 3) * 2, acc[nd8][2 * i], acc[nd8][2 * i + 1]);
      }
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
  // dqI: fragment rows 0..7 (e = 0, 1) are the indexer heads
#pragma unroll
  for (int i = 0; i < kDQPerWarp; ++i) {
    const int blk = warp + i * NW;
    const int h = lane >> 2;
    if (blk >= kDQB || h >= H_I) continue;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int col = blk * 16 + j * 8 + (lane & 3) * 2;
      TIn* dst = dqI + ((int64_t)row * H_I + h) * DI + col;
      dst[0] = from_f32<TIn>(dqf[i][j][0]);
      dst[1] = from_f32<TIn>(dqf[i][j][1]);
    }
  }
}

template <typename TIn, int D, int NW, int DI>
static cudaError_t launch_kl_bwd_t(const KLBwdArgs& a, cudaStream_t stream) {
  constexpr int kStride = AttnSmem<D>::kStride;
  constexpr int kThreads = NW * 32;
  constexpr int kHK = 8 * kKeys;
  const size_t smem = (size_t)(NW * 16 + 2 * kKeys) * kStride * 2 +
                      ((size_t)2 * kKeys * (DI + 8) + 16 * (DI + 8) + 16 * (kKeys + 8)) * 2 +
                      ((size_t)8 * DI + 8 + NW * kKeys + kHK + kKeys + (kHK > 2 * kThreads ? kHK : 2 * kThreads)) * 4;
  auto kern = indexer_kl_bwd_kernel<TIn, D, NW, DI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  constexpr float kLog2e = 1.4426950408889634f;
  kern<<<a.T_cap, kThreads, smem, stream>>>(
      static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k_cmp), static_cast<const TIn*>(a.qI),
      static_cast<const TIn*>(a.w), static_cast<const TIn*>(a.kI), a.idx, a.k_pad, a.lse_cmp, a.student_lse, a.cu,
      a.cu_cmp, a.B,
      a.H, a.H_I, a.r, a.scale * kLog2e, a.grad_scale, static_cast<TIn*>(a.dqI), static_cast<TIn*>(a.dw), a.dkI,
      a.status, a.pos0);
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
  if (indexer_kl_bwd_tc_supported(a, fp32)) return launch_indexer_kl_bwd_tc(a, stream);
  if (indexer_kl_bwd_sparse_tc_supported(a, fp32)) return launch_indexer_kl_bwd_sparse_tc(a, stream);
  cudaError_t err = cudaMemsetAsync(a.dkI, 0, (size_t)a.n_cmp_cap * a.d_I * 4, stream);
  if (err != cudaSuccess) return err;
  return fp32 ? kl_bwd_dims<float>(a, stream) : kl_bwd_dims<__nv_bfloat16>(a, stream);
}

}  // namespace csa
