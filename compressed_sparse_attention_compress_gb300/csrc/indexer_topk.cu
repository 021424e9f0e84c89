// indexer_topk.cu -- lightning-indexer scoring fused with the per-query top-k.
//
// "DeepSeek-V4 Attention Training Systems": §3 (indexer logit i_{t,j}; here
// sum_h w[t,h] ReLU(qI[t,h,:] . kI[j,:])), §4 (causal visibility of completed
// groups, reset at sample boundaries), §8 and §8.2 ("indexer scoring and radix
// top-k"; causal offsets, ragged lengths, fixed top-k capacity, alignment
// padding and local-to-global id lowering are part of correctness), §8.1
// (top-k list padded to an alignment).
//
// One CTA owns G consecutive queries of one sequence.  Their G*H_I indexer
// query rows form the A operand of a tensor-core tile (mma.sync m16n8k16 bf16,
// fp32 accumulate); 64-entry tiles of the sequence's compressed indexer keys
// stream through shared memory (cp.async, double buffered).  The epilogue
// applies ReLU and the head weights, sums the heads with warp shuffles and
// keeps every score in shared memory as an order-preserving 32-bit key: the
// score matrix never leaves the SM.  Selection is an exact radix select over
// those keys (11 + 11 + 10 bit digits, warp-aggregated shared-memory
// histograms), followed by an ordered compaction that emits the selected
// entries in ascending index order (ties at the threshold: smaller index
// first), lowered to global compressed rows and padded with -1.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sm80.cuh"

namespace csa {

namespace {

constexpr int kThreads = 128;
constexpr int kTileN = 64;        // indexer keys per tile
constexpr int kMaxRows = 64;      // G * H_I query rows per CTA
constexpr int kBins = 2048;

__device__ __forceinline__ uint32_t order_key(float v) {
  if (v == 0.f) v = 0.f;  // -0 and +0 are the same score
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one value per thread (kThreads threads).
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int base = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int x = s_warp[w];
    if (w < warp) base += x;
    total += x;
  }
  __syncthreads();
  return base + incl - v;
}

}  // namespace

template <typename TIn, int DI>
__global__ void __launch_bounds__(kThreads)
indexer_topk_kernel(const TIn* __restrict__ qI, const TIn* __restrict__ w, const TIn* __restrict__ kI,
                    const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_cmp, int B, int H_I,
                    int G, int max_vis, int r, int topk, int k_pad, int32_t* __restrict__ idx, int* status,
                    const int32_t* __restrict__ pos0) {
  constexpr int kAStride = DI + 8;
  extern __shared__ __align__(128) uint8_t smem[];
  const int vstride = (max_vis + 3) & ~3;                                              // 16-byte rows
  uint32_t* sKey = reinterpret_cast<uint32_t*>(smem);                                  // [G][vstride]
  __nv_bfloat16* sA = reinterpret_cast<__nv_bfloat16*>(sKey + (size_t)G * vstride);    // [64][kAStride]
  __nv_bfloat16* sB = sA + kMaxRows * kAStride;                                        // [2][64][kAStride]
  uint32_t* sHist = reinterpret_cast<uint32_t*>(sB + 2 * kTileN * kAStride);           // [kBins]
  float* sW = reinterpret_cast<float*>(sHist + kBins);                                 // [64]
  __shared__ int s_b, s_q0, s_nq;
  __shared__ int s_warp[kThreads / 32];
  __shared__ uint32_t s_digit;
  __shared__ int s_need;
  __shared__ int s_cnt[2][kThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    int c = blockIdx.x, b = -1, L = 0;
    for (int bb = 0; bb < B; ++bb) {
      L = __ldg(cu + bb + 1) - __ldg(cu + bb);
      if (L < 0) { raise_status(status, CSA_ERR_DEVICE_BOUNDS); L = 0; }
      // the last query of the sequence sees (L + p0) / r entries (p0: position of its first row)
      const int pp = pos0 ? __ldg(pos0 + bb) : 0;
      if ((L + pp) / r > max_vis) { raise_status(status, CSA_ERR_DEVICE_BOUNDS); L = 0; }
      const int nch = (L + G - 1) / G;
      if (c < nch) { b = bb; break; }
      c -= nch;
    }
    s_b = b;
    s_q0 = c * G;
    s_nq = b >= 0 ? min(G, L - c * G) : 0;
  }
  __syncthreads();
  const int b = s_b;
  if (b < 0) return;
  const int q0 = s_q0, nq = s_nq;
  const int seq0 = __ldg(cu + b);
  const int cmp0 = __ldg(cu_cmp + b);
  const int p0 = pos0 ? __ldg(pos0 + b) : 0;  // position of the sequence's first row here
  const int n_b = (__ldg(cu + b + 1) - seq0 + p0) / r;
  const int rows = G * H_I;
  const int mtiles = (rows + 15) / 16;
  const int vis_last = min((q0 + nq + p0) / r, max_vis);  // visible entries of the chunk's last query
  const int ntiles = (vis_last + kTileN - 1) / kTileN;

  // A operand: indexer query rows (g, h) -> row g*H_I + h; zero past nq.
  for (int i = tid; i < kMaxRows * (DI / 8); i += kThreads) {
    const int rr = i / (DI / 8), c = i - rr * (DI / 8);
    const int g = rr / H_I, h = rr - g * H_I;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (rr < rows && g < nq) v = Load8<TIn>::run(qI + ((int64_t)(seq0 + q0 + g) * H_I + h) * DI + c * 8);
    *reinterpret_cast<uint4*>(sA + rr * kAStride + c * 8) = v;
  }
  for (int i = tid; i < kMaxRows; i += kThreads) {
    const int g = i / H_I, h = i - g * H_I;
    sW[i] = (i < rows && g < nq) ? to_f32(w[(int64_t)(seq0 + q0 + g) * H_I + h]) : 0.f;
  }

  auto issue = [&](int it, int buf) {
    for (int i = tid; i < kTileN * (DI / 8); i += kThreads) {
      const int k = i / (DI / 8), c = i - k * (DI / 8);
      const int j = it * kTileN + k;
      __nv_bfloat16* dst = sB + (buf * kTileN + k) * kAStride + c * 8;
      const bool ok = j < n_b;
      if constexpr (sizeof(TIn) == 2) {
        cp_async_16_zfill(smem_u32(dst), kI + (int64_t)(cmp0 + (ok ? j : 0)) * DI + c * 8, ok);
      } else {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (ok) v = Load8<TIn>::run(kI + (int64_t)(cmp0 + j) * DI + c * 8);
        *reinterpret_cast<uint4*>(dst) = v;
      }
    }
  };

  // ---- scores of every visible entry into shared memory ----
  if (ntiles > 0) issue(0, 0);
  cp_async_commit();
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntiles) issue(it + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const __nv_bfloat16* tB = sB + buf * kTileN * kAStride;
    for (int mt = 0; mt < mtiles; ++mt) {
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < DI / 16; ++kk) {
        uint32_t a[4], bq[4];
        ldmatrix_x4(smem_u32(sA + (mt * 16 + (lane & 15)) * kAStride + kk * 16 + (lane >> 4) * 8), a[0], a[1],
                    a[2], a[3]);
        const int key = warp * 16 + (lane & 7) + (lane >> 4) * 8;
        ldmatrix_x4(smem_u32(tB + key * kAStride + kk * 16 + ((lane >> 3) & 1) * 8), bq[0], bq[1], bq[2],
                    bq[3]);
        mma_bf16_16816(c[0], a, bq);
        mma_bf16_16816(c[1], a, bq + 2);
      }
      // w * ReLU, then sum over the H_I consecutive rows of each query
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rr = mt * 16 + (lane >> 2) + (e >> 1) * 8;
          float v = sW[rr] * fmaxf(c[nt][e], 0.f);
          for (int o = 4; o < 4 * H_I; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          c[nt][e] = v;
        }
      }
      if (((lane >> 2) % H_I) == 0) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int rr = mt * 16 + (lane >> 2) + (e >> 1) * 8;
            const int g = rr / H_I;
            const int j = it * kTileN + warp * 16 + nt * 8 + (lane & 3) * 2 + (e & 1);
            if (rr < rows && g < nq && j < max_vis) sKey[(size_t)g * vstride + j] = order_key(c[nt][e]);
          }
        }
      }
    }
    __syncthreads();
  }

  // ---- per query: exact radix select + ordered compaction ----
  for (int g = 0; g < nq; ++g) {
    const int t = q0 + g;
    const int64_t orow = (int64_t)(seq0 + t) * k_pad;
    const int n = min((t + p0 + 1) / r, max_vis);
    const int m = min(topk, n);
    const uint32_t* keys = sKey + (size_t)g * vstride;
    uint32_t thr = 0;
    int need_eq = 0;
    const bool all = n <= topk;
    if (!all) {
      uint32_t prefix = 0, pmask = 0;
      int need = m;
      for (int round = 0; round < 3; ++round) {
        const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
        const int bits = round == 2 ? 10 : 11;
        const uint32_t dmask = (1u << bits) - 1u;
        for (int i = tid; i < kBins; i += kThreads) sHist[i] = 0;
        __syncthreads();
        for (int jb = warp * 32; jb < n; jb += kThreads) {
          const int j = jb + lane;
          const uint32_t key = j < n ? keys[j] : 0u;
          const bool ok = j < n && (key & pmask) == prefix;
          const uint32_t act = __ballot_sync(0xffffffffu, ok);
          if (ok) {
            const uint32_t dg = (key >> shift) & dmask;
            const uint32_t peers = __match_any_sync(act, dg);
            if (lane == __ffs(peers) - 1) atomicAdd(&sHist[dg], (uint32_t)__popc(peers));
          }
        }
        __syncthreads();
        // thread tid owns bins [top - 16(tid+1), top - 16 tid) counted from the top
        constexpr int kPer = kBins / kThreads;
        const int nb = (int)dmask + 1;
        const int hi_bin = nb - 1 - tid * kPer;  // highest bin this thread owns
        int local = 0;
        for (int k = 0; k < kPer; ++k) {
          const int bin = hi_bin - k;
          if (bin >= 0) local += (int)sHist[bin];
        }
        int total;
        const int above = block_excl_scan(local, s_warp, total);
        if (above < need && need <= above + local) {
          int cum = above;
          for (int k = 0; k < kPer; ++k) {
            const int bin = hi_bin - k;
            if (bin < 0) break;
            const int hcount = (int)sHist[bin];
            if (need <= cum + hcount) {
              s_digit = (uint32_t)bin;
              s_need = need - cum;
              break;
            }
            cum += hcount;
          }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        pmask |= dmask << shift;
        need = s_need;
        __syncthreads();
      }
      thr = prefix;
      need_eq = need;
    }
    // ordered compaction: warp w scans the contiguous range [w*seg, (w+1)*seg)
    const int seg = ((n + kThreads - 1) / kThreads) * 32;
    const int j_lo = warp * seg, j_hi = min(n, j_lo + seg);
    int gt = 0, eq = 0;
    for (int jb = j_lo; jb < j_hi; jb += 32) {
      const int j = jb + lane;
      const uint32_t key = j < j_hi ? keys[j] : 0u;
      gt += __popc(__ballot_sync(0xffffffffu, j < j_hi && (all || key > thr)));
      eq += __popc(__ballot_sync(0xffffffffu, j < j_hi && !all && key == thr));
    }
    if (lane == 0) { s_cnt[0][warp] = gt; s_cnt[1][warp] = eq; }
    __syncthreads();
    int gt_before = 0, eq_before = 0;
    for (int ww = 0; ww < warp; ++ww) { gt_before += s_cnt[0][ww]; eq_before += s_cnt[1][ww]; }
    for (int jb = j_lo; jb < j_hi; jb += 32) {
      const int j = jb + lane;
      const uint32_t key = j < j_hi ? keys[j] : 0u;
      const bool fgt = j < j_hi && (all || key > thr);
      const bool feq = j < j_hi && !all && key == thr;
      const uint32_t bgt = __ballot_sync(0xffffffffu, fgt);
      const uint32_t beq = __ballot_sync(0xffffffffu, feq);
      const uint32_t below = (1u << lane) - 1u;
      const int my_gt = gt_before + __popc(bgt & below);
      const int my_eq = eq_before + __popc(beq & below);
      if (fgt || (feq && my_eq < need_eq)) {
        const int pos = my_gt + min(my_eq, need_eq);
        idx[orow + pos] = cmp0 + j;
      }
      gt_before += __popc(bgt);
      eq_before += __popc(beq);
    }
    for (int i = m + tid; i < k_pad; i += kThreads) idx[orow + i] = -1;
    __syncthreads();
  }
}

// idx rows of capacity padding (rows >= cu[B]) are all -1.
__global__ void topk_fill_capacity_kernel(const int32_t* __restrict__ cu, int B, int T_cap, int k_pad,
                                          int32_t* __restrict__ idx) {
  const int64_t start = (int64_t)__ldg(cu + B) * k_pad;
  const int64_t end = (int64_t)T_cap * k_pad;
  for (int64_t i = start + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < end;
       i += (int64_t)gridDim.x * blockDim.x)
    idx[i] = -1;
}

static int topk_group(int H_I, int max_vis) {
  int G = (96 * 1024) / (4 * (max_vis > 0 ? max_vis : 1));
  if (G > kMaxRows / H_I) G = kMaxRows / H_I;
  if (G < 1) G = 1;
  return G;
}

static size_t topk_smem(int G, int max_vis, int DI) {
  return (size_t)G * ((max_vis + 3) & ~3) * 4 + (size_t)(kMaxRows + 2 * kTileN) * (DI + 8) * 2 + kBins * 4 + kMaxRows * 4;
}

bool indexer_topk_supported(int H_I, int d_I, int max_vis, int k_pad, int in_bytes) {
  (void)in_bytes;
  (void)k_pad;
  const int G = topk_group(H_I, max_vis);
  return topk_smem(G, max_vis, d_I) <= 220 * 1024;
}

template <typename TIn, int DI>
static cudaError_t launch_topk_t(const void* qI, const void* w, const void* kI, const int32_t* cu,
                                 const int32_t* cu_cmp, int B, int T_cap, int max_vis, int H_I, int r,
                                 int topk, int k_pad, int32_t* idx, int* status, cudaStream_t stream,
                                 const int32_t* pos0) {
  const int G = topk_group(H_I, max_vis);
  const size_t smem = topk_smem(G, max_vis, DI);
  auto kern = indexer_topk_kernel<TIn, DI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long grid = (long long)T_cap / G + B + 1;
  if (T_cap > 0) {
    kern<<<(unsigned)grid, kThreads, smem, stream>>>(static_cast<const TIn*>(qI), static_cast<const TIn*>(w),
                                                     static_cast<const TIn*>(kI), cu, cu_cmp, B, H_I, G, max_vis,
                                                     r, topk, k_pad, idx, status, pos0);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    topk_fill_capacity_kernel<<<152, 256, 0, stream>>>(cu, B, T_cap, k_pad, idx);
  }
  return cudaGetLastError();
}

cudaError_t launch_indexer_topk_fp8_full(const uint8_t* qI, const float* qs, const void* w, const uint8_t* kI,
                                         const float* ks, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap,
                                         int max_vis, int r, int topk, int k_pad, int32_t* idx, int* status,
                                         cudaStream_t stream, const int32_t* pos0, int cmp_rows) {
  cudaError_t err = launch_indexer_topk_fp8(qI, qs, w, kI, ks, cu, cu_cmp, B, T_cap, max_vis, r, topk, k_pad, idx,
                                            status, stream, pos0, cmp_rows);
  if (err != cudaSuccess || T_cap <= 0) return err;
  topk_fill_capacity_kernel<<<152, 256, 0, stream>>>(cu, B, T_cap, k_pad, idx);
  return cudaGetLastError();
}

cudaError_t launch_indexer_topk(const void* qI, const void* w, const void* kI, const int32_t* cu,
                                const int32_t* cu_cmp, int B, int T_cap, int max_vis, int H_I, int d_I, int r,
                                int topk, int k_pad, bool fp32, int32_t* idx, int* status, cudaStream_t stream,
                                const int32_t* pos0, int cmp_rows) {
  // indexer 8 heads x 64 dims in bf16 scores on tcgen05 with TMA-fed tiles
  if (indexer_topk_tc_supported(H_I, d_I, max_vis, fp32)) {
    cudaError_t err = launch_indexer_topk_tc(qI, w, kI, cu, cu_cmp, B, T_cap, max_vis, r, topk, k_pad, idx, status,
                                             stream, pos0, cmp_rows);
    if (err != cudaSuccess || T_cap <= 0) return err;
    topk_fill_capacity_kernel<<<152, 256, 0, stream>>>(cu, B, T_cap, k_pad, idx);
    return cudaGetLastError();
  }
  if (fp32) {
    if (d_I == 32)
      return launch_topk_t<float, 32>(qI, w, kI, cu, cu_cmp, B, T_cap, max_vis, H_I, r, topk, k_pad, idx, status,
                                      stream, pos0);
    return launch_topk_t<float, 64>(qI, w, kI, cu, cu_cmp, B, T_cap, max_vis, H_I, r, topk, k_pad, idx, status,
                                    stream, pos0);
  }
  if (d_I == 32)
    return launch_topk_t<__nv_bfloat16, 32>(qI, w, kI, cu, cu_cmp, B, T_cap, max_vis, H_I, r, topk, k_pad, idx,
                                            status, stream, pos0);
  return launch_topk_t<__nv_bfloat16, 64>(qI, w, kI, cu, cu_cmp, B, T_cap, max_vis, H_I, r, topk, k_pad, idx,
                                          status, stream, pos0);
}

}  // namespace csa
