// attention.cu -- selected (CSA), HCA and window-only attention forward.
//
// "DeepSeek-V4 Attention Training Systems": §2 phase table (top-k compressed
// entries + local window; HCA reads every completed ratio-128 entry plus the
// window; window-only layers have no compressor), §8.2 (selected MQA attention
// over a flat global index list returning output and LSE; compressed ids are
// combined with window ids), §9 (FP32 attention sink, FP32 softmax).
//
// One CTA per query row; its warps split the query heads (16 heads per warp)
// and share every gathered key tile (MQA: one KV head).  The candidate list is
// the compressed part (idx row / every visible entry / nothing) followed by
// the window part; each part is cut into tiles of 64 keys.  A tile's rows are
// resolved to packed row numbers first (validity and visibility checks happen
// here), then gathered into shared memory with 16-byte cp.async copies, two
// tiles in flight.  S = Q K^T and O += P V run on the tensor cores
// (mma.sync m16n8k16 bf16, fp32 accumulate) with an online softmax in the
// exp2 domain; the compressed-only normaliser (lse_cmp) is taken when the
// compressed part ends.
// Precision: the normalisers are sums of the bf16-rounded weights that enter
// the P V products (the output is a convex combination of the value rows with
// the weights used); the reference is the exact running maximum.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sm80.cuh"
#include "tile_sm80.cuh"

namespace csa {


template <typename TIn, typename TOut, int D, int NW>
__global__ void __launch_bounds__(NW * 32)
attention_kernel(int kind, const TIn* __restrict__ q, const TIn* __restrict__ k_cmp,
                 const TIn* __restrict__ v_cmp, const TIn* __restrict__ k_raw,
                 const TIn* __restrict__ v_raw, const int32_t* __restrict__ idx, int k_pad,
                 const float* __restrict__ sink, const int32_t* __restrict__ cu,
                 const int32_t* __restrict__ cu_cmp, int B, int H, int r, int window, float scale_log2,
                 TOut* __restrict__ out, float* __restrict__ lse, float* __restrict__ lse_cmp,
                 int* status,
                 const int32_t* __restrict__ pos0) {
  constexpr int kStride = AttnSmem<D>::kStride;
  constexpr int kRows = NW * 16;
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sK = sQ + kRows * kStride;           // [2][kKeys][kStride]
  __nv_bfloat16* sV = sK + 2 * kKeys * kStride;       // [2][kKeys][kStride] (separate V only)
  __shared__ int s_rows[2][kKeys];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int b = owner_sequence(cu, B, row);
  const bool separate_v = (v_cmp != nullptr) || (v_raw != nullptr);
  const TIn* vc = v_cmp ? v_cmp : k_cmp;
  const TIn* vr = v_raw ? v_raw : k_raw;

  if (b < 0) {  // capacity row
    for (int i = tid; i < H * D; i += NW * 32) out[(int64_t)row * H * D + i] = from_f32<TOut>(0.f);
    for (int h = tid; h < H; h += NW * 32) {
      lse[(int64_t)row * H + h] = -INFINITY;
      if (lse_cmp) lse_cmp[(int64_t)row * H + h] = -INFINITY;
    }
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

  // Q rows of this query (heads >= H are zero).
  for (int i = tid; i < kRows * (D / 8); i += NW * 32) {
    const int h = i / (D / 8), c = i - h * (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h < H) v = Load8<TIn>::run(q + ((int64_t)row * H + h) * D + c * 8);
    *reinterpret_cast<uint4*>(sQ + h * kStride + c * 8) = v;
  }

  const int cmp_limit = (kind == kAttnWindow) ? 0 : __ldg(cu_cmp + B);  // packed compressed rows
  const int raw_limit = __ldg(cu + B);                                    // packed raw rows
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

  float o_acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float lsec[2] = {-INFINITY, -INFINITY};  // compressed-only log2 normaliser

  if (ntiles > 0) {
    resolve(0, 0);
    __syncthreads();
    issue(0, 0);
  }
  cp_async_commit();

  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    if (it == n_ctiles) {  // compressed part finished: snapshot its normaliser
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float l = l_run[i];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        lsec[i] = l > 0.f ? m_run[i] + __log2f(l) : -INFINITY;
      }
    }
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

    // S = Q K^T for this warp's 16 heads x 64 keys.
    float s[8][4];
    qk_tile<D>(sQ, tK, warp, lane, s);
    // mask + scale (log2 domain) + row max
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = n * 8 + (lane & 3) * 2 + (e & 1);
        const float v = s_rows[buf][key] >= 0 ? s[n][e] * scale_log2 : -INFINITY;
        s[n][e] = v;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
      }
    }
    float alpha[2], muse[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 1));
      tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 2));
      const float mnew = fmaxf(m_run[i], tmax[i]);
      muse[i] = mnew == -INFINITY ? 0.f : mnew;
      alpha[i] = exp2f(m_run[i] - muse[i]);
      m_run[i] = mnew;
      l_run[i] *= alpha[i];
    }
    uint32_t pa[4][4];  // P as A fragments, one per 16-key step
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float p0 = exp2f(s[n][0] - muse[0]), p1 = exp2f(s[n][1] - muse[0]);
      const float p2 = exp2f(s[n][2] - muse[1]), p3 = exp2f(s[n][3] - muse[1]);
      const uint32_t a01 = pack_bf16x2(p0, p1), a23 = pack_bf16x2(p2, p3);
      pa[n >> 1][(n & 1) * 2 + 0] = a01;
      pa[n >> 1][(n & 1) * 2 + 1] = a23;
      l_run[0] += bf16_lo(a01) + bf16_hi(a01);  // the sums are of the weights as written
      l_run[1] += bf16_lo(a23) + bf16_hi(a23);
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o_acc[i][0] *= alpha[0];
      o_acc[i][1] *= alpha[0];
      o_acc[i][2] *= alpha[1];
      o_acc[i][3] *= alpha[1];
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int nd = 0; nd < D / 16; ++nd) {
        uint32_t bv[4];
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int col = nd * 16 + (lane >> 4) * 8;
        ldmatrix_x4_trans(smem_u32(tV + key * kStride + col), bv[0], bv[1], bv[2], bv[3]);
        mma_bf16_16816(o_acc[2 * nd], pa[kk], bv);
        mma_bf16_16816(o_acc[2 * nd + 1], pa[kk], bv + 2);
      }
    }
    __syncthreads();
  }
  if (ntiles == n_ctiles) {  // no window tile ran (cannot happen: the window holds t)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float l = l_run[i];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      lsec[i] = l > 0.f ? m_run[i] + __log2f(l) : -INFINITY;
    }
  }

  // finalise: quad-reduce l, add the sink, normalise, store
  constexpr float kLn2 = 0.6931471805599453f;
  constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float l = l_run[i];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int h = warp * 16 + (lane >> 2) + i * 8;
    float m = m_run[i];
    float corr = 1.f;
    if (sink != nullptr && h < H) {
      const float s2 = __ldg(sink + h) * kLog2e;
      const float mf = fmaxf(m, s2);
      corr = exp2f(m - mf);
      l = l * corr + exp2f(s2 - mf);
      m = mf;
    }
    const float inv = l > 0.f ? corr / l : 0.f;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      o_acc[nd][2 * i] *= inv;
      o_acc[nd][2 * i + 1] *= inv;
    }
    if (h < H && (lane & 3) == 0) {
      lse[(int64_t)row * H + h] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
      if (lse_cmp) lse_cmp[(int64_t)row * H + h] = lsec[i] * kLn2;
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int h = warp * 16 + (lane >> 2) + i * 8;
    if (h >= H) continue;
    TOut* orow = out + ((int64_t)row * H + h) * D;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const int col = nd * 8 + (lane & 3) * 2;
      orow[col] = from_f32<TOut>(o_acc[nd][2 * i]);
      orow[col + 1] = from_f32<TOut>(o_acc[nd][2 * i + 1]);
    }
  }
}

template <typename TIn, typename TOut, int D, int NW>
static cudaError_t launch_attention_t(AttnKind kind, const AttnArgs& a, cudaStream_t stream) {
  constexpr int kStride = AttnSmem<D>::kStride;
  const bool separate_v = a.v_cmp != nullptr || a.v_raw != nullptr;
  const size_t smem = (size_t)(NW * 16 + (separate_v ? 4 : 2) * kKeys) * kStride * 2;
  auto kern = attention_kernel<TIn, TOut, D, NW>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (a.T_cap <= 0) return cudaSuccess;
  constexpr float kLog2e = 1.4426950408889634f;
  kern<<<a.T_cap, NW * 32, smem, stream>>>(
      (int)kind, static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k_cmp), static_cast<const TIn*>(a.v_cmp),
      static_cast<const TIn*>(a.k_raw), static_cast<const TIn*>(a.v_raw), a.idx, a.k_pad, a.sink, a.cu,
      a.cu_cmp, a.B, a.H, a.r, a.window, a.scale * kLog2e, static_cast<TOut*>(a.out), a.lse, a.lse_cmp,
      a.status, a.pos0);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int D>
static cudaError_t dispatch_heads(AttnKind kind, const AttnArgs& a, cudaStream_t stream) {
  switch ((a.H + 15) / 16) {
    case 1: return launch_attention_t<TIn, TOut, D, 1>(kind, a, stream);
    case 2: return launch_attention_t<TIn, TOut, D, 2>(kind, a, stream);
    case 4: return launch_attention_t<TIn, TOut, D, 4>(kind, a, stream);
    case 8: return launch_attention_t<TIn, TOut, D, 8>(kind, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attention(AttnKind kind, const AttnArgs& a, bool fp32, cudaStream_t stream) {
  // 64 heads x 128 dims in bf16 (every workload of the pages) run on tcgen05;
  // other head counts / dims and float32 I/O use the warp-level kernel above.
  if (attention_ws_supported(a, fp32)) return launch_attention_ws(kind, a, stream);
  if (attention_tc_supported(a, fp32)) return launch_attention_tc(kind, a, stream);
  if (fp32) {
    if (a.d == 64) return dispatch_heads<float, float, 64>(kind, a, stream);
    return dispatch_heads<float, float, 128>(kind, a, stream);
  }
  if (a.d == 64) return dispatch_heads<__nv_bfloat16, __nv_bfloat16, 64>(kind, a, stream);
  return dispatch_heads<__nv_bfloat16, __nv_bfloat16, 128>(kind, a, stream);
}

}  // namespace csa
