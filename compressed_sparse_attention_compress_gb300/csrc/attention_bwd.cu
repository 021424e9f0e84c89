// attention_bwd.cu -- backward of the selected (CSA), HCA and window-only
// attention: Q, K/V and attention-sink gradients from the saved output and LSE.
//
// "DeepSeek-V4 Attention Training Systems": §8.2 (the main attention backward
// "consumes saved output/LSE and produces Q, KV, and attention-sink gradients
// without materializing a dense attention matrix"), §9 (FP32 sink, FP32
// softmax math).  With p_i = exp(s_i - lse) the forward weights of candidate i
// (s_i = scale q.K_i), D = dout.o, and the upstream gradient dout:
//   ds_i = p_i (dout.V_i - D),  dq = scale sum_i ds_i K_i,
//   dK_i += scale ds_i q,  dV_i += p_i dout,  dsink -= exp(sink - lse) D.
//
// Three launches.  attn_bwd_delta_kernel: D per (row, head), one warp each.
// attention_bwd_kernel: one CTA per query row, the forward's candidate tiles
// of 64 keys gathered the same way (cp.async, two tiles in flight); per tile
// the warps (16 heads each) recompute S = Q K^T and dP = dO V^T on mma.sync,
// form P and scale*dS, accumulate dq = (scale dS) K in registers (written once
// at the end), then -- after a block barrier that publishes P and dS as bf16
// tiles -- each warp takes 16 of the 64 keys and forms that key block's
// gradient summed over every head, dK = (scale dS)^T Q and dV = P^T dO, as
// mma.sync products over the heads, added to the float32 key / value gradient
// rows with vector red.global.add (the rows stay in L2: the compressed rows
// are shared by every query that selected them, a raw row by the W queries
// whose window holds it).  attn_bwd_dsink_kernel: the sink gradient, one CTA
// per head, fixed summation order.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sm80.cuh"
#include "tile_sm80.cuh"

namespace csa {

namespace {

constexpr int kPStride = kKeys + 8;  // bf16 elements per row of the P / dS tiles (16 B pad)

__device__ __forceinline__ void red_add_v2(float* p, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};\n" ::"l"(p), "f"(a), "f"(b) : "memory");
}

template <typename T> struct Load4;
template <> struct Load4<__nv_bfloat16> {
  static __device__ __forceinline__ float4 run(const __nv_bfloat16* p) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
  }
};
template <> struct Load4<float> {
  static __device__ __forceinline__ float4 run(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
};

}  // namespace

// delta[row, h] = sum_c dout[row,h,c] * out[row,h,c]; 0 for capacity rows.
template <typename TIn>
__global__ void __launch_bounds__(256)
attn_bwd_delta_kernel(const TIn* __restrict__ out, const TIn* __restrict__ dout, const int32_t* __restrict__ cu,
                      int B, int T_cap, int H, int D, float* __restrict__ delta) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= (int64_t)T_cap * H) return;
  const int64_t row = w / H;
  float acc = 0.f;
  if (row < __ldg(cu + B)) {
    for (int c = lane * 4; c < D; c += 128) {
      const float4 o = Load4<TIn>::run(out + w * D + c), g = Load4<TIn>::run(dout + w * D + c);
      acc = fmaf(o.x, g.x, fmaf(o.y, g.y, fmaf(o.z, g.z, fmaf(o.w, g.w, acc))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) delta[w] = acc;
}

// dsink[h] = -sum_rows exp(sink[h] - lse[row,h]) * delta[row,h]; one CTA per head.
__global__ void __launch_bounds__(256)
attn_bwd_dsink_kernel(const float* __restrict__ sink, const float* __restrict__ lse,
                      const float* __restrict__ delta, const int32_t* __restrict__ cu, int B, int H,
                      float* __restrict__ dsink) {
  __shared__ float s_part[8];
  const int h = blockIdx.x;
  const int T = __ldg(cu + B);
  const float sk = __ldg(sink + h);
  float acc = 0.f;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const float l = __ldg(lse + (int64_t)t * H + h);
    if (l > -INFINITY) acc = fmaf(expf(sk - l), __ldg(delta + (int64_t)t * H + h), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += s_part[i];
    dsink[h] = -s;
  }
}

template <typename TIn, typename TOut, int D, int NW>
__global__ void __launch_bounds__(NW * 32)
attention_bwd_kernel(int kind, const TIn* __restrict__ q, const TIn* __restrict__ k_cmp,
                     const TIn* __restrict__ v_cmp, const TIn* __restrict__ k_raw, const TIn* __restrict__ v_raw,
                     const int32_t* __restrict__ idx, int k_pad, const int32_t* __restrict__ cu,
                     const int32_t* __restrict__ cu_cmp, int B, int H, int r, int window, float scale,
                     float scale_log2, const float* __restrict__ lse, const float* __restrict__ delta,
                     const TIn* __restrict__ dout, TOut* __restrict__ dq, float* __restrict__ dk_cmp,
                     float* __restrict__ dv_cmp, float* __restrict__ dk_raw, float* __restrict__ dv_raw,
                     int* status,
                     const int32_t* __restrict__ pos0) {
  constexpr int kStride = AttnSmem<D>::kStride;
  constexpr int kRows = NW * 16;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sG = sQ + kRows * kStride;            // dO rows
  __nv_bfloat16* sP = sG + kRows * kStride;            // [kRows][kPStride] P (bf16)
  __nv_bfloat16* sDS = sP + kRows * kPStride;          // [kRows][kPStride] scale * dS (bf16)
  __nv_bfloat16* sK = sDS + kRows * kPStride;          // [2][kKeys][kStride]
  __nv_bfloat16* sV = sK + 2 * kKeys * kStride;        // [2][kKeys][kStride] (separate V only)
  __shared__ int s_rows[2][kKeys];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int b = owner_sequence(cu, B, row);
  const bool separate_v = (v_cmp != nullptr) || (v_raw != nullptr);
  const TIn* vc = v_cmp ? v_cmp : k_cmp;
  const TIn* vr = v_raw ? v_raw : k_raw;

  if (b < 0) {  // capacity row: no candidates, dq = 0
    for (int i = tid; i < H * D; i += NW * 32) dq[(int64_t)row * H * D + i] = from_f32<TOut>(0.f);
    return;
  }
  const int seq0 = __ldg(cu + b);
  const int t = row - seq0;
  const int p0 = pos0 ? __ldg(pos0 + b) : 0;  // position of the sequence's first row here
  const int nvis = (kind == kAttnWindow || r <= 0) ? 0 : (t + p0 + 1) / r;
  const int cmp0 = (kind == kAttnWindow) ? 0 : __ldg(cu_cmp + b);
  const int w0 = max(0, t - window + 1);
  const int n_win = t - w0 + 1;
  const int n_cslots = kind == kAttnCSA ? k_pad : (kind == kAttnHCA ? nvis : 0);
  const int n_ctiles = (n_cslots + kKeys - 1) / kKeys;
  const int ntiles = n_ctiles + (n_win + kKeys - 1) / kKeys;

  // Q and dO rows of this query (heads >= H are zero).
  for (int i = tid; i < kRows * (D / 8); i += NW * 32) {
    const int h = i / (D / 8), c = i - h * (D / 8);
    uint4 vq = make_uint4(0, 0, 0, 0), vg = make_uint4(0, 0, 0, 0);
    if (h < H) {
      vq = Load8<TIn>::run(q + ((int64_t)row * H + h) * D + c * 8);
      vg = Load8<TIn>::run(dout + ((int64_t)row * H + h) * D + c * 8);
    }
    *reinterpret_cast<uint4*>(sQ + h * kStride + c * 8) = vq;
    *reinterpret_cast<uint4*>(sG + h * kStride + c * 8) = vg;
  }
  // this thread's two heads (rows lane/4 and lane/4 + 8 of the warp's 16)
  float lse2[2], dl[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int h = warp * 16 + (lane >> 2) + i * 8;
    lse2[i] = h < H ? __ldg(lse + (int64_t)row * H + h) * kLog2e : INFINITY;  // padded heads: p = 0
    dl[i] = h < H ? __ldg(delta + (int64_t)row * H + h) : 0.f;
  }

  const int cmp_limit = (kind == kAttnWindow) ? 0 : __ldg(cu_cmp + B);
  const int raw_limit = __ldg(cu + B);
  auto resolve = [&](int it, int buf) {
    for (int kk = tid; kk < kKeys; kk += NW * 32) {
      int rr = -1;
      if (it < n_ctiles) {
        const int slot = it * kKeys + kk;
        if (kind == kAttnCSA) {
          if (slot < k_pad) {
            const int g = __ldg(idx + (int64_t)row * k_pad + slot);
            if (g >= 0) {
              if (g < cmp0 || g >= cmp0 + nvis) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
              else rr = g;
            }
          }
        } else if (slot < nvis) {
          rr = cmp0 + slot;
        }
      } else {
        const int wi = (it - n_ctiles) * kKeys + kk;
        if (wi < n_win) rr = seq0 + w0 + wi;
      }
      s_rows[buf][kk] = rr;
    }
  };
  auto issue = [&](int it, int buf) {
    const bool cmp = it < n_ctiles;
    gather_tile<TIn, D>(cmp ? k_cmp : k_raw, cmp ? vc : vr, separate_v, s_rows[buf], cmp ? cmp_limit : raw_limit,
                        sK + buf * kKeys * kStride, sV + buf * kKeys * kStride, tid, NW * 32);
  };

  float dq_acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dq_acc[i][0] = dq_acc[i][1] = dq_acc[i][2] = dq_acc[i][3] = 0.f;

  if (ntiles > 0) {
    resolve(0, 0);
    __syncthreads();
    issue(0, 0);
  }
  cp_async_commit();

  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntiles) {
      resolve(it + 1, buf ^ 1);
      __syncthreads();
      issue(it + 1, buf ^ 1);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const __nv_bfloat16* tK = sK + buf * kKeys * kStride;
    const __nv_bfloat16* tV = separate_v ? sV + buf * kKeys * kStride : tK;
    const bool cmp_tile = it < n_ctiles;

    // S = Q K^T and dP = dO V^T for this warp's 16 heads x 64 keys
    float s[8][4], dp[8][4];
    qk_tile<D>(sQ, tK, warp, lane, s);
    qk_tile<D>(sG, tV, warp, lane, dp);
    uint32_t pa[4][4], da[4][4];  // P and scale*dS as A fragments, one per 16-key step
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      float p[4], g[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = n * 8 + (lane & 3) * 2 + (e & 1);
        p[e] = s_rows[buf][key] >= 0 ? exp2f(fmaf(s[n][e], scale_log2, -lse2[e >> 1])) : 0.f;
        g[e] = p[e] * (dp[n][e] - dl[e >> 1]) * scale;
      }
      pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16x2(p[0], p[1]);
      pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16x2(p[2], p[3]);
      da[n >> 1][(n & 1) * 2 + 0] = pack_bf16x2(g[0], g[1]);
      da[n >> 1][(n & 1) * 2 + 1] = pack_bf16x2(g[2], g[3]);
      // publish the tiles for the key-side products: rows = heads, columns = keys
      const int h0 = warp * 16 + (lane >> 2), key0 = n * 8 + (lane & 3) * 2;
      *reinterpret_cast<uint32_t*>(sP + h0 * kPStride + key0) = pa[n >> 1][(n & 1) * 2 + 0];
      *reinterpret_cast<uint32_t*>(sP + (h0 + 8) * kPStride + key0) = pa[n >> 1][(n & 1) * 2 + 1];
      *reinterpret_cast<uint32_t*>(sDS + h0 * kPStride + key0) = da[n >> 1][(n & 1) * 2 + 0];
      *reinterpret_cast<uint32_t*>(sDS + (h0 + 8) * kPStride + key0) = da[n >> 1][(n & 1) * 2 + 1];
    }
    // dq += (scale dS) K
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int nd = 0; nd < D / 16; ++nd) {
        uint32_t bk[4];
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int col = nd * 16 + (lane >> 4) * 8;
        ldmatrix_x4_trans(smem_u32(tK + key * kStride + col), bk[0], bk[1], bk[2], bk[3]);
        mma_bf16_16816(dq_acc[2 * nd], da[kk], bk);
        mma_bf16_16816(dq_acc[2 * nd + 1], da[kk], bk + 2);
      }
    }
    __syncthreads();  // P and dS of every head are in shared memory

    // key blocks of 16: dK = (scale dS)^T Q and dV = P^T dO over all heads
    float* dk_dst = cmp_tile ? dk_cmp : dk_raw;
    float* dv_dst = separate_v ? (cmp_tile ? dv_cmp : dv_raw) : dk_dst;
    for (int kg = warp; kg < kKeys / 16; kg += NW) {
      const int m0 = kg * 16;
      float acc[D / 8][4];
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        if (pass == 0 || separate_v) {
#pragma unroll
          for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        }
        const __nv_bfloat16* tA = pass == 0 ? sDS : sP;   // [heads][keys]
        const __nv_bfloat16* tB = pass == 0 ? sQ : sG;    // [heads][d]
#pragma unroll
        for (int kh = 0; kh < kRows / 16; ++kh) {
          uint32_t a[4];
          const int mi = lane >> 3;
          ldmatrix_x4_trans(smem_u32(tA + (kh * 16 + (mi >> 1) * 8 + (lane & 7)) * kPStride + m0 + (mi & 1) * 8),
                            a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nd = 0; nd < D / 16; ++nd) {
            uint32_t bq[4];
            const int hr = kh * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int col = nd * 16 + (lane >> 4) * 8;
            ldmatrix_x4_trans(smem_u32(tB + hr * kStride + col), bq[0], bq[1], bq[2], bq[3]);
            mma_bf16_16816(acc[2 * nd], a, bq);
            mma_bf16_16816(acc[2 * nd + 1], a, bq + 2);
          }
        }
        if (pass == 1 || separate_v) {
          float* dst = pass == 0 ? dk_dst : dv_dst;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int rr = s_rows[buf][m0 + (lane >> 2) + i * 8];
            if (rr < 0) continue;
#pragma unroll
            for (int nd8 = 0; nd8 < D / 8; ++nd8)
              red_add_v2(dst + (int64_t)rr * D + nd8 * 8 + (lane & 3) * 2, acc[nd8][2 * i], acc[nd8][2 * i + 1]);
          }
        }
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int h = warp * 16 + (lane >> 2) + i * 8;
    if (h >= H) continue;
    TOut* grow = dq + ((int64_t)row * H + h) * D;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const int col = nd * 8 + (lane & 3) * 2;
      grow[col] = from_f32<TOut>(dq_acc[nd][2 * i]);
      grow[col + 1] = from_f32<TOut>(dq_acc[nd][2 * i + 1]);
    }
  }
}

template <typename TIn, typename TOut, int D, int NW>
static cudaError_t launch_bwd_t(AttnKind kind, const AttnBwdArgs& a, cudaStream_t stream) {
  constexpr int kStride = AttnSmem<D>::kStride;
  const bool separate_v = a.v_cmp != nullptr || a.v_raw != nullptr;
  const size_t smem = ((size_t)(2 * NW * 16 + (separate_v ? 4 : 2) * kKeys) * kStride +
                       (size_t)2 * NW * 16 * kPStride) * 2;
  auto kern = attention_bwd_kernel<TIn, TOut, D, NW>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  constexpr float kLog2e = 1.4426950408889634f;
  kern<<<a.T_cap, NW * 32, smem, stream>>>(
      (int)kind, static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k_cmp), static_cast<const TIn*>(a.v_cmp),
      static_cast<const TIn*>(a.k_raw), static_cast<const TIn*>(a.v_raw), a.idx, a.k_pad, a.cu, a.cu_cmp, a.B, a.H,
      a.r, a.window, a.scale, a.scale * kLog2e, a.lse, a.delta, static_cast<const TIn*>(a.dout),
      static_cast<TOut*>(a.dq), a.dk_cmp, a.dv_cmp, a.dk_raw, a.dv_raw, a.status, a.pos0);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int D>
static cudaError_t bwd_dispatch_heads(AttnKind kind, const AttnBwdArgs& a, cudaStream_t stream) {
  switch ((a.H + 15) / 16) {
    case 1: return launch_bwd_t<TIn, TOut, D, 1>(kind, a, stream);
    case 2: return launch_bwd_t<TIn, TOut, D, 2>(kind, a, stream);
    case 4: return launch_bwd_t<TIn, TOut, D, 4>(kind, a, stream);
    case 8: return launch_bwd_t<TIn, TOut, D, 8>(kind, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename TIn>
static cudaError_t launch_bwd_all(AttnKind kind, const AttnBwdArgs& a, cudaStream_t stream) {
  // gradient rows are accumulated: start from zero
  const size_t d = (size_t)a.d;
  cudaError_t err = cudaSuccess;
  if (a.dk_cmp && (err = cudaMemsetAsync(a.dk_cmp, 0, (size_t)a.n_cmp_cap * d * 4, stream)) != cudaSuccess) return err;
  if (a.dv_cmp && (err = cudaMemsetAsync(a.dv_cmp, 0, (size_t)a.n_cmp_cap * d * 4, stream)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(a.dk_raw, 0, (size_t)a.T_cap * d * 4, stream)) != cudaSuccess) return err;
  if (a.dv_raw && (err = cudaMemsetAsync(a.dv_raw, 0, (size_t)a.T_cap * d * 4, stream)) != cudaSuccess) return err;
  const long long warps = (long long)a.T_cap * a.H;
  attn_bwd_delta_kernel<TIn><<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(
      static_cast<const TIn*>(a.out), static_cast<const TIn*>(a.dout), a.cu, a.B, a.T_cap, a.H, a.d, a.delta);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  // 64 heads x 128 dims in bf16 with K = V run on tcgen05; other shapes on the warp-level kernel
  if (attention_bwd_tc_supported(a, sizeof(TIn) == 4)) err = launch_attention_bwd_tc(kind, a, stream);
  else if (a.d == 64) err = bwd_dispatch_heads<TIn, TIn, 64>(kind, a, stream);
  else err = bwd_dispatch_heads<TIn, TIn, 128>(kind, a, stream);
  if (err != cudaSuccess) return err;
  if (a.sink && a.dsink) {
    attn_bwd_dsink_kernel<<<a.H, 256, 0, stream>>>(a.sink, a.lse, a.delta, a.cu, a.B, a.H, a.dsink);
    err = cudaGetLastError();
  }
  return err;
}

cudaError_t launch_attention_bwd(AttnKind kind, const AttnBwdArgs& a, bool fp32, cudaStream_t stream) {
  if (a.T_cap <= 0) return cudaSuccess;
  return fp32 ? launch_bwd_all<float>(kind, a, stream) : launch_bwd_all<__nv_bfloat16>(kind, a, stream);
}

}  // namespace csa
