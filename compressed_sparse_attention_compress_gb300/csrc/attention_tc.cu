// attention_tc.cu -- selected / HCA / window attention forward on the 5th-gen
// tensor cores (tcgen05, accumulators in tensor memory), 64 heads x 128 dims.
//
// "DeepSeek-V4 Attention Training Systems": §2 phase table, §8.2 (selected MQA
// attention over a flat global index list returning output and LSE; compressed
// ids combined with window ids), §9 (FP32 sink, FP32 softmax).
//
// Every query has its own key list (its top-k entries + its window), shared by
// its 64 heads (one KV head).  A 64-row MMA would leave half of the tensor core
// idle, so the tile is transposed: the 128 gathered keys are the M dimension.
//   S^T[key, h]  = K[key, :] . Q[h, :]        M=128 keys, N=64 heads, K=128 dims
//   O^T[dim, h] += V^T[dim, key] P^T[key, h]  M=128 dims, N=64 heads, K=128 keys
// Both accumulators live in tensor memory (64 + 64 columns).  The gathered tile
// (128 rows x 256 B, 128-byte swizzle) is the K-major A operand of the first
// MMA and, read the other way, the MN-major A operand of the second.
//
// Softmax.  Thread k of the 4 warps owns tensor-memory lane k = key k and reads
// that key's 64 head scores.  The per-head maximum runs across lanes, so it is
// kept lazily: the running reference m_h changes only when a score exceeds it
// by more than 2^8 (checked with one block vote per tile); then the tile's
// column maxima are taken with warp max-reductions, and the per-thread partial
// sums and the O^T columns are rescaled.  P^T is written to shared memory as
// bf16 rows of 64 heads (one swizzled 128-byte row per key) for the second MMA.
// Per-head sums stay per thread until the end of the query (warp butterfly +
// shared memory reduction).
//
// Pipelining: the gather of tile i+1 (cp.async, zero-filled for missing keys)
// runs during the softmax of tile i; PV(i) and QK(i+1) are issued together;
// two CTAs share an SM.  Compressed tiles with no valid entry are skipped.
// Precision: as in the warp-specialised kernel, the normalisers are sums of
// the bf16-rounded weights that enter P^T, and the reference is the exact
// maximum while a query has seen fewer than kExactKeys keys.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace csa {

namespace {

constexpr int kTK = 128;       // keys per tile (M of the first MMA)
constexpr int kNH = 64;        // heads (N of both MMAs)
constexpr int kDim = 128;      // head dim
constexpr int kThr = 128;      // one thread per tensor-memory lane
constexpr float kTau = 8.f;    // lazy-max slack, log2 units
constexpr int kExactKeys = 32;  // exact maximum until this many keys were seen

constexpr uint32_t kQRegion = kNH * 128;      // 8 KB: 64 rows x 64 dims
constexpr uint32_t kTileRegion = kTK * 128;   // 16 KB: 128 rows x 64 dims
constexpr uint32_t kTileBytes = 2 * kTileRegion;
constexpr uint32_t kQOff = 0;
constexpr uint32_t kStage0 = 2 * kQRegion;    // 16 KB

template <bool SEPV>
struct Layout {
  static constexpr uint32_t kStageBytes = (SEPV ? 2 : 1) * kTileBytes;
  static constexpr uint32_t kPOff = kStage0 + 2 * kStageBytes;
  static constexpr uint32_t kBytes = kPOff + kTK * 128;  // + P^T (16 KB)
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order-preserving float <-> int for integer max reductions.
__device__ __forceinline__ int ord_of(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float float_of(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF); }

// Sum 64 per-thread values over the 32 lanes of a warp; afterwards lane l
// holds the sums of entries 2l and 2l+1 in v[0], v[1].
__device__ __forceinline__ void warp_sum64(float (&v)[64], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int half = 32 >> step;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < half) {
        const float send = upper ? v[j] : v[j + half];
        const float keep = upper ? v[j + half] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
}

}  // namespace

template <bool SEPV>
__global__ void __launch_bounds__(kThr, 2)
attention_tc_kernel(int kind, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cmp,
                    const __nv_bfloat16* __restrict__ v_cmp, const __nv_bfloat16* __restrict__ k_raw,
                    const __nv_bfloat16* __restrict__ v_raw, const int32_t* __restrict__ idx, int k_pad,
                    const float* __restrict__ sink, const int32_t* __restrict__ cu,
                    const int32_t* __restrict__ cu_cmp, int B, int T_cap, int r, int window, float scale_log2,
                    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, float* __restrict__ lse_cmp,
                    int* status,
                    const int32_t* __restrict__ pos0) {
  using L = Layout<SEPV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_bar[3];  // 0: S ready, 1: O (PV) done, 2: the issuer's last commit
  __shared__ int s_rows[2][kTK];
  __shared__ __align__(16) float s_m[kNH];
  __shared__ float s_alpha[kNH], s_inv[kNH];
  __shared__ int s_wmax[4][kNH];
  __shared__ float s_lsum[4][kNH];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_s = smem_u32(&s_bar[0]), bar_o = smem_u32(&s_bar[1]);

  if (warp == 0) {
    tc::tmem_alloc(smem_u32(&s_tmem), 128);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(smem_u32(&s_bar[2]), 1);
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t t_s = tmem;                           // S^T: columns 0..63
  const uint32_t t_o = tmem + kNH;                     // O^T: columns 64..127
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  constexpr uint32_t kIdescQK = tc::idesc_bf16(kTK, kNH, 0, 0);
  constexpr uint32_t kIdescPV = tc::idesc_bf16(kDim, kNH, 1, 1);
  uint32_t ph_s = 0, ph_o = 0;  // mbarrier phases consumed so far

  const int cmp_limit = kind == kAttnWindow ? 0 : __ldg(cu_cmp + B);
  const int raw_limit = __ldg(cu + B);
  const __nv_bfloat16* vc = SEPV ? v_cmp : k_cmp;
  const __nv_bfloat16* vr = SEPV ? v_raw : k_raw;

  // longest queries first: rows are handed out from the end of the buffer
  for (int qi = blockIdx.x; qi < T_cap; qi += gridDim.x) {
    const int row = T_cap - 1 - qi;
    const int b = owner_sequence(cu, B, row);
    if (b < 0) {
      for (int i = tid; i < kNH * kDim; i += kThr) out[(int64_t)row * kNH * kDim + i] = __float2bfloat16(0.f);
      if (tid < kNH) {
        lse[(int64_t)row * kNH + tid] = -INFINITY;
        if (lse_cmp) lse_cmp[(int64_t)row * kNH + tid] = -INFINITY;
      }
      continue;
    }
    const int seq0 = __ldg(cu + b);
    const int t = row - seq0;
    const int p0 = pos0 ? __ldg(pos0 + b) : 0;  // position of the sequence's first row here
    const int nvis = (kind == kAttnWindow || r <= 0) ? 0 : (t + p0 + 1) / r;
    const int cmp0 = kind == kAttnWindow ? 0 : __ldg(cu_cmp + b);
    const int w0 = max(0, t - window + 1);
    const int n_win = t - w0 + 1;
    const int n_cslots = kind == kAttnCSA ? k_pad : (kind == kAttnHCA ? nvis : 0);
    const int n_ctiles = (n_cslots + kTK - 1) / kTK;
    const int ntiles = n_ctiles + (n_win + kTK - 1) / kTK;

    // this thread's index-list slot of tile `it`, loaded one tile ahead of its use
    int pre_it = -1, pre_g = -1;
    auto prefetch = [&](int it) {
      const int slot = it * kTK + tid;
      if (kind == kAttnCSA && it < n_ctiles && slot < k_pad) {
        asm volatile("ld.global.nc.b32 %0, [%1];\n" : "=r"(pre_g) : "l"(idx + (int64_t)row * k_pad + slot));
        pre_it = it;
      }
    };
    // resolve the rows of tile `it` into s_rows[buf]; true if any is valid
    auto resolve = [&](int it, int buf) -> bool {
      int rr = -1;
      if (it < n_ctiles) {
        const int slot = it * kTK + tid;
        if (kind == kAttnCSA) {
          if (slot < k_pad) {
            const int g = pre_it == it ? pre_g : __ldg(idx + (int64_t)row * k_pad + slot);
            if (g >= 0) {
              if (g < cmp0 || g >= cmp0 + nvis || g >= cmp_limit) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
              else rr = g;
            }
          }
        } else if (slot < nvis) {
          rr = cmp0 + slot;
        }
      } else {
        const int wi = (it - n_ctiles) * kTK + tid;
        if (wi < n_win && seq0 + w0 + wi < raw_limit) rr = seq0 + w0 + wi;
      }
      s_rows[buf][tid] = rr;
      prefetch(it + 1);
      return __syncthreads_or(rr >= 0) != 0;
    };
    // first tile index >= it with a valid key (window tiles always have one)
    auto next_tile = [&](int it, int buf) -> int {
      while (it < ntiles && !resolve(it, buf)) ++it;
      return it;
    };
    auto gather = [&](int it, int buf) {
      const bool cmpt = it < n_ctiles;
      const __nv_bfloat16* ks = cmpt ? k_cmp : k_raw;
      const __nv_bfloat16* vs = cmpt ? vc : vr;
      const uint32_t kb = base + kStage0 + buf * L::kStageBytes;
#pragma unroll 4
      for (int i = tid; i < kTK * 16; i += kThr) {
        const int key = i >> 4, c = i & 15;
        const int rr = s_rows[buf][key];
        const uint32_t dst = kb + (c >> 3) * kTileRegion + tc::sw128_offset(key, c & 7);
        const int64_t src = (int64_t)(rr < 0 ? 0 : rr) * kDim + c * 8;
        cp_async_16_zfill(dst, ks + src, rr >= 0);
        if constexpr (SEPV) cp_async_16_zfill(dst + kTileBytes, vs + src, rr >= 0);
      }
      cp_async_commit();
    };
    auto issue_qk = [&](int buf) {
      const uint32_t kb = base + kStage0 + buf * L::kStageBytes;
#pragma unroll
      for (int ks = 0; ks < kDim / 16; ++ks) {
        const uint64_t a = tc::smem_desc_sw128(kb + (ks >> 2) * kTileRegion + (ks & 3) * 32, 16, 1024);
        const uint64_t bq = tc::smem_desc_sw128(base + kQOff + (ks >> 2) * kQRegion + (ks & 3) * 32, 16, 1024);
        tc::mma_bf16(t_s, a, bq, kIdescQK, ks > 0 ? 1u : 0u);
      }
      tc::mma_commit(bar_s);
    };
    auto issue_pv = [&](int buf, bool first) {
      const uint32_t vb = base + kStage0 + buf * L::kStageBytes + (SEPV ? kTileBytes : 0);
#pragma unroll
      for (int ks = 0; ks < kTK / 16; ++ks) {
        const uint64_t a = tc::smem_desc_sw128(vb + ks * 2048, kTileRegion, 1024);
        // N = 64 heads is one 128-byte atom: the M/N-direction offset is never used
        const uint64_t bp = tc::smem_desc_sw128(base + L::kPOff + ks * 2048, 1024, 1024);
        tc::mma_bf16(t_o, a, bp, kIdescPV, (first && ks == 0) ? 0u : 1u);
      }
      tc::mma_commit(bar_o);
    };
    // every thread waits; false (for all threads) if any of them ran out of time
    auto wait = [&](uint32_t bar, uint32_t& ph) -> bool {
      const bool ok = mbar_wait_bounded(bar, ph & 1u, status);
      ++ph;
      return __syncthreads_or(!ok) == 0;
    };
    // block-wide per-head sums of the per-thread partials l (destroys l)
    auto head_sums = [&](float (&l)[64]) {
      warp_sum64(l, lane);
      s_lsum[warp][2 * lane] = l[0];
      s_lsum[warp][2 * lane + 1] = l[1];
      __syncthreads();
    };

    // ---- Q (swizzled K-major, two 64-dim regions) and the first tile ----
    for (int i = tid; i < kNH * 16; i += kThr) {
      const int h = i >> 4, c = i & 15;
      cp_async_16(base + kQOff + (c >> 3) * kQRegion + tc::sw128_offset(h, c & 7),
                  q + ((int64_t)row * kNH + h) * kDim + c * 8);
    }
    if (tid < kNH) s_m[tid] = -INFINITY;
    int cur = next_tile(0, 0);
    int buf = 0;
    gather(cur, buf);
    cp_async_wait<0>();
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      issue_qk(buf);
    }

    float l_part[kNH];
#pragma unroll
    for (int h = 0; h < kNH; ++h) l_part[h] = 0.f;
    bool have_o = false, snap = false;
    int seen = 0;  // keys of this query in the tiles before this one

    bool aborted = false;
    while (cur < ntiles) {
      // rows of the next tile (s_rows[buf ^ 1] is no longer read), then its gather
      // into buffer buf ^ 1 once the previous tile's PV has finished reading it
      const int nxt = (cur + 1 < ntiles) ? next_tile(cur + 1, buf ^ 1) : ntiles;
      if (have_o && !wait(bar_o, ph_o)) { aborted = true; break; }
      if (nxt < ntiles) gather(nxt, buf ^ 1);

      if (!snap && cur >= n_ctiles) {  // compressed candidates done: their normaliser
        snap = true;
        if (lse_cmp != nullptr) {
          float tmp[kNH];
#pragma unroll
          for (int h = 0; h < kNH; ++h) tmp[h] = l_part[h];
          head_sums(tmp);
          if (tid < kNH) {
            const float l = s_lsum[0][tid] + s_lsum[1][tid] + s_lsum[2][tid] + s_lsum[3][tid];
            lse_cmp[(int64_t)row * kNH + tid] = l > 0.f ? (s_m[tid] + __log2f(l)) * 0.6931471805599453f : -INFINITY;
          }
          __syncthreads();
        }
      }

      if (!wait(bar_s, ph_s)) { aborted = true; break; }
      tc::fence_after_sync();

      // ---- softmax of tile `cur`: this thread = key (tid) ----
      // t_h = s_h * scale*log2(e) - m_h, the log2 weight relative to the running
      // reference; a block vote decides whether any t_h exceeds the slack.
      const bool valid = s_rows[buf][tid] >= 0;
      float t[kNH];
      auto load_t = [&]() {
        uint32_t rs[32];
        tc::tmem_ld32_sync(t_s + lane_off, rs);
#pragma unroll
        for (int j = 0; j < 32; ++j) t[j] = __uint_as_float(rs[j]);
        tc::tmem_ld32_sync(t_s + lane_off + 32, rs);
#pragma unroll
        for (int j = 0; j < 32; ++j) t[32 + j] = __uint_as_float(rs[j]);
      };
      auto to_log2_weights = [&]() -> float {  // t <- s*c - m; returns max_h t
        float ex = -INFINITY;
#pragma unroll
        for (int h4 = 0; h4 < kNH / 4; ++h4) {
          const float4 m4 = reinterpret_cast<const float4*>(s_m)[h4];
          t[4 * h4 + 0] = fmaf(t[4 * h4 + 0], scale_log2, -m4.x);
          t[4 * h4 + 1] = fmaf(t[4 * h4 + 1], scale_log2, -m4.y);
          t[4 * h4 + 2] = fmaf(t[4 * h4 + 2], scale_log2, -m4.z);
          t[4 * h4 + 3] = fmaf(t[4 * h4 + 3], scale_log2, -m4.w);
          ex = fmaxf(ex, fmaxf(fmaxf(t[4 * h4 + 0], t[4 * h4 + 1]), fmaxf(t[4 * h4 + 2], t[4 * h4 + 3])));
        }
        return ex;
      };
      load_t();
      float excess = -INFINITY;
      if (valid) excess = to_log2_weights();  // m = -inf (first tile) gives +inf
      // the reference is the exact running maximum while the query has seen fewer
      // than kExactKeys keys (with few candidates one key can carry most of the
      // weight: its P^T weight is then exactly 1, free of bf16 rounding), and lags by
      // up to kTau after that
      if (__syncthreads_or(excess > (seen < kExactKeys ? 0.f : kTau))) {
        // new reference: the tile's per-head column maxima (warp max-reductions)
        load_t();
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          const float xh = valid ? t[h] * scale_log2 : -INFINITY;
          const int v = __reduce_max_sync(0xffffffffu, ord_of(xh));
          if (lane == 0) s_wmax[warp][h] = v;
        }
        __syncthreads();
        if (tid < kNH) {
          const float mo = s_m[tid];
          float mn = mo;
#pragma unroll
          for (int w = 0; w < 4; ++w) mn = fmaxf(mn, float_of(s_wmax[w][tid]));
          s_alpha[tid] = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
          s_m[tid] = mn;
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < kNH; ++h) l_part[h] *= s_alpha[h];
        if (have_o) {  // O^T row `tid` (one head dim), columns = heads
#pragma unroll
          for (int c0 = 0; c0 < kNH; c0 += 16) {
            uint32_t ro[16];
            tc::tmem_ld16_sync(t_o + lane_off + c0, ro);
#pragma unroll
            for (int j = 0; j < 16; ++j) ro[j] = __float_as_uint(__uint_as_float(ro[j]) * s_alpha[c0 + j]);
            tc::tmem_st16(t_o + lane_off + c0, ro);
          }
          tc::tmem_wait_st();
        }
        if (valid) to_log2_weights();
      }
      // P^T row of this key: 64 heads -> 8 swizzled 16-byte chunks (zeros for a missing key)
      {
        const uint32_t prow = base + L::kPOff;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t pk[4] = {0u, 0u, 0u, 0u};
          if (valid) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int h = c * 8 + 2 * j;
              pk[j] = pack_bf16x2(ex2(t[h]), ex2(t[h + 1]));
              l_part[h] += bf16_lo(pk[j]);  // the sums are of the weights as written
              l_part[h + 1] += bf16_hi(pk[j]);
            }
          }
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + tc::sw128_offset(tid, c)),
                       "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                       : "memory");
        }
      }
      tc::fence_before_sync();
      tc::fence_proxy_async_smem();
      cp_async_wait<0>();           // next tile's gather has landed
      tc::fence_proxy_async_smem();
      seen += __syncthreads_count(valid);
      if (tid == 0) {
        tc::fence_after_sync();
        issue_pv(buf, !have_o);
        if (nxt < ntiles) issue_qk(buf ^ 1);
      }
      have_o = true;
      cur = nxt;
      buf ^= 1;
    }
    if (!aborted && have_o && !wait(bar_o, ph_o)) aborted = true;
    if (aborted) break;  // uniform: the status word says why
    tc::fence_after_sync();

    // ---- epilogue: per-head normaliser, sink, O / l, LSE ----
    head_sums(l_part);
    if (tid < kNH) {
      float l = s_lsum[0][tid] + s_lsum[1][tid] + s_lsum[2][tid] + s_lsum[3][tid];
      float m = s_m[tid];
      float corr = 1.f;
      if (sink != nullptr) {
        const float s2 = __ldg(sink + tid) * 1.4426950408889634f;
        const float mf = fmaxf(m, s2);
        corr = (m == -INFINITY) ? 0.f : ex2(m - mf);
        l = l * corr + ex2(s2 - mf);
        m = mf;
      }
      s_inv[tid] = l > 0.f ? corr / l : 0.f;
      lse[(int64_t)row * kNH + tid] = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    {
      __nv_bfloat16* orow = out + (int64_t)row * kNH * kDim + tid;  // this thread's head dim
#pragma unroll
      for (int c0 = 0; c0 < kNH; c0 += 32) {
        uint32_t ro[32];
        tc::tmem_ld32_sync(t_o + lane_off + c0, ro);
#pragma unroll
        for (int j = 0; j < 32; ++j) orow[(c0 + j) * kDim] = __float2bfloat16(__uint_as_float(ro[j]) * s_inv[c0 + j]);
      }
    }
    tc::fence_before_sync();
    __syncthreads();
  }

  // leave no copy or MMA in flight and give the tensor memory back
  cp_async_wait<0>();
  if (tid == 0) {  // thread 0 issued every MMA: their completion, also after an abort
    tc::mma_commit(smem_u32(&s_bar[2]));
    mbar_wait_bounded(smem_u32(&s_bar[2]), 0, status);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

bool attention_tc_supported(const AttnArgs& a, bool fp32) {
  return !fp32 && a.H == kNH && a.d == kDim;
}

template <bool SEPV>
static cudaError_t launch_tc_t(AttnKind kind, const AttnArgs& a, cudaStream_t stream) {
  using L = Layout<SEPV>;
  const size_t smem = L::kBytes + 2048;  // + alignment slack
  auto kern = attention_tc_kernel<SEPV>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (a.T_cap <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_sm = SEPV ? 1 : 2;
  const int grid = a.T_cap < sms * per_sm ? a.T_cap : sms * per_sm;
  constexpr float kLog2e = 1.4426950408889634f;
  kern<<<grid, kThr, smem, stream>>>(
      (int)kind, static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_cmp),
      static_cast<const __nv_bfloat16*>(a.v_cmp), static_cast<const __nv_bfloat16*>(a.k_raw),
      static_cast<const __nv_bfloat16*>(a.v_raw), a.idx, a.k_pad, a.sink, a.cu, a.cu_cmp, a.B, a.T_cap, a.r,
      a.window, a.scale * kLog2e, static_cast<__nv_bfloat16*>(a.out), a.lse, a.lse_cmp, a.status, a.pos0);
  return cudaGetLastError();
}

cudaError_t launch_attention_tc(AttnKind kind, const AttnArgs& a, cudaStream_t stream) {
  const bool sepv = a.v_cmp != nullptr || a.v_raw != nullptr;
  return sepv ? launch_tc_t<true>(kind, a, stream) : launch_tc_t<false>(kind, a, stream);
}

}  // namespace csa
