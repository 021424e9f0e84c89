// indexer_topk_tc.cu -- lightning-indexer scoring on tcgen05 tensor cores with
// TMA-fed key tiles, fused with the exact per-query top-k (indexer 8 heads x
// 64 dims, bf16).
//
// "DeepSeek-V4 Attention Training Systems": §3 (indexer logit i_{t,j}; here
// sum_h w[t,h] ReLU(qI[t,h,:] . kI[j,:])), §4 (causal visibility of completed
// groups, reset at sample boundaries), §8 / §8.2 ("indexer scoring and radix
// top-k": causal offsets, ragged lengths, fixed top-k capacity, alignment
// padding and local-to-global id lowering), §8.1 (top-k padding).
//
// One CTA takes a block of G consecutive queries of one sequence (G = 4, or 2
// for very long sequences).  Their visible entries are a prefix of the
// sequence's compressed rows, so the key tiles (128 entries x 64 dims) are
// shared: a TMA warp streams them through a 2- or 4-stage pipeline, an MMA
// warp computes I^T = kI qI^T (M = 128 entries, N = G x 8 query-heads) into a
// four-deep ring of tensor-memory tiles, and the compute warps turn each entry's
// head scores into sum_h w ReLU(.) for their queries, store it in shared
// memory (float) and track each query's score range.  No score reaches global
// memory.  Then each warpgroup selects one query at a time, exactly:
//   * a histogram of value-linear buckets over the query's [min, max] score
//     (monotone in the score, so every entry in a bucket above the one that
//     holds the k-th largest is selected, and only that bucket needs the
//     exact order);
//   * one pass counts, per warp segment, the entries above that bucket and
//     lists the bucket's entries (order-preserving 32-bit key, index);
//   * one warp finds the exact k-th largest key among them bit by bit and the
//     number of entries equal to it still selected (ties: smaller index first);
//     when the bucket holds more entries than the list, an exact 8-bit radix
//     select over all the keys takes its place;
//   * an ordered compaction writes the selected entries in ascending index
//     order as global compressed rows, -1 padded.
// Blocks whose queries all see at most k entries select everything without
// scoring.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace csa {

#ifdef CSA_TOPK_PROFILE
// Profiling build only: cycles per site, summed over compute warps.
__device__ unsigned long long g_topk_prof[16];
#define TK_T0(v) const long long v = clock64()
#define TK_ADD(site, v) \
  do {                  \
    if (lane == 0) atomicAdd(&g_topk_prof[site], (unsigned long long)(clock64() - (v))); \
  } while (0)
#define TK_CNT(site) \
  do {               \
    if (lane == 0) atomicAdd(&g_topk_prof[site], 1ull); \
  } while (0)
#else
#define TK_T0(v)
#define TK_ADD(site, v)
#define TK_CNT(site)
#endif

namespace {

constexpr int kHI = 8, kDI = 64;
constexpr int kTK = 128;                 // entries per tile
// selection: value-linear buckets of one query's score range, then the list of
// the entries in the threshold's bucket (key, index), in one 4 KB region per
// selecting warpgroup
constexpr int kSelBins = 1024;
constexpr int kSelBytes = 4096;
constexpr int kCand = kSelBytes / 8;
constexpr uint32_t kTileBytes = kTK * 128;  // 16 KB
constexpr int kDBufs = 4;                   // score tiles in tensor memory (32 columns each)
constexpr uint32_t kQIOff = 0;              // up to 32 rows x 128 B
constexpr uint32_t kStageOff = 4096;

// Two shapes: 16 compute warps and a 4-stage ring, one CTA per SM; or 8 compute
// warps and a 2-stage ring, two CTAs per SM (one CTA selects while the other
// scores).
template <int CW>
struct TopkCfg {
  static constexpr int kStages = CW == 8 ? 2 : 4;
  static constexpr int kCtasPerSm = CW == 8 ? 2 : 1;
  static constexpr int kThreads = 32 * CW + 64;
  static constexpr uint32_t kKeysOff = kStageOff + kStages * kTileBytes;  // scores start here
};

__device__ __forceinline__ uint32_t order_key(float v) {
  if (v == 0.f) v = 0.f;  // -0 and +0 are the same score
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float of an order-preserving key (the inverse of order_key).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp: the need-th largest order key among the c candidates (key, entry
// index) of `cand`, searched bit by bit below the bits every candidate shares;
// then, per warp segment u (entry index / seg, four segments), the candidates
// above it (g[u]) and equal to it (e[u]).  thr: that key; need_eq: how many of
// the equal ones are still selected.  Every lane gets every result.
__device__ __forceinline__ void resolve_candidates(const uint2* cand, int c, int need, int seg, int lane,
                                                   uint32_t& thr, int& need_eq, int (&g)[4], int (&e)[4]) {
  const bool regs = c <= 64;  // the common case: the keys stay in registers
  const uint32_t r0 = (regs && lane < c) ? cand[lane].x : 0u;
  const uint32_t r1 = (regs && lane + 32 < c) ? cand[lane + 32].x : 0u;
  uint32_t kand = 0xFFFFFFFFu, kor = 0u;
  for (int i = lane; i < c; i += 32) {
    const uint32_t k = cand[i].x;
    kand &= k;
    kor |= k;
  }
  kand = __reduce_and_sync(0xffffffffu, kand);
  kor = __reduce_or_sync(0xffffffffu, kor);
  const uint32_t diff = kand ^ kor;
  uint32_t pre = kand;
  if (diff != 0u) {
    const int top = 31 - __clz(diff);
    pre = kand & ~((2u << top) - 1u);  // the shared leading bits (top = 31: none)
    for (int bit = top; bit >= 0; --bit) {
      const uint32_t trial = pre | (1u << bit);
      int cnt = 0;
      if (regs) {
        cnt = (r0 >= trial ? 1 : 0) + (r1 >= trial ? 1 : 0);  // empty slots hold 0 < trial
      } else {
        for (int i = lane; i < c; i += 32) cnt += cand[i].x >= trial ? 1 : 0;
      }
      if (__reduce_add_sync(0xffffffffu, cnt) >= need) pre = trial;
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) g[u] = e[u] = 0;
  for (int i = lane; i < c; i += 32) {
    const uint2 cd = cand[i];
    const int w = (int)cd.y / seg;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      g[u] += (w == u && cd.x > pre) ? 1 : 0;
      e[u] += (w == u && cd.x == pre) ? 1 : 0;
    }
  }
  int gsum = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    g[u] = __reduce_add_sync(0xffffffffu, g[u]);
    e[u] = __reduce_add_sync(0xffffffffu, e[u]);
    gsum += g[u];
  }
  thr = pre;
  need_eq = need - gsum;
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

struct QBlock {
  int q0, nq, seq0, cmp0, p0, nvis_max, ntiles;
  bool score;  // some query sees more than k entries
};

__device__ __forceinline__ int total_qblocks(const int32_t* __restrict__ cu, int B, int G) {
  int n = 0;
  for (int bb = 0; bb < B; ++bb) n += (max(0, __ldg(cu + bb + 1) - __ldg(cu + bb)) + G - 1) / G;
  return n;
}

// Block k counted from the end of the buffer (latest queries, most entries, first).
__device__ __forceinline__ bool qblock_of(const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_cmp, int B,
                                          int r, int G, int topk, int max_vis, int total, int k, QBlock& o,
                                          const int32_t* __restrict__ pos0) {
  int c = total - 1 - k;
  for (int bb = 0; bb < B; ++bb) {
    const int L = max(0, __ldg(cu + bb + 1) - __ldg(cu + bb));
    const int nb = (L + G - 1) / G;
    if (c < nb) {
      o.q0 = c * G;
      o.nq = min(G, L - c * G);
      o.seq0 = __ldg(cu + bb);
      o.cmp0 = __ldg(cu_cmp + bb);
      o.p0 = pos0 ? __ldg(pos0 + bb) : 0;  // position of the sequence's first row here
      o.nvis_max = min((o.q0 + o.nq + o.p0) / r, max_vis);
      o.score = o.nvis_max > topk;
      o.ntiles = o.score ? (o.nvis_max + kTK - 1) / kTK : 0;
      return true;
    }
    c -= nb;
  }
  return false;
}

}  // namespace

// kFp8: qI and kI are E4M3 codes with per-row power-of-two scales (qs per
// query head, ks per compressed row); the scores are then
// ks[j] * sum_h (w_h qs_h) ReLU(codes dot), the same as the dequantised
// operands give since the scales are positive.
template <int G, int CW, bool kFp8>
__global__ void __launch_bounds__(TopkCfg<CW>::kThreads, TopkCfg<CW>::kCtasPerSm)
indexer_topk_tc_kernel(const __grid_constant__ CUtensorMap map_qi, const __grid_constant__ CUtensorMap map_ki,
                       const __nv_bfloat16* __restrict__ w, const float* __restrict__ qs,
                       const float* __restrict__ ks, const int32_t* __restrict__ cu,
                       const int32_t* __restrict__ cu_cmp, int B, int r, int topk, int k_pad, int max_vis,
                       int32_t* __restrict__ idx, int* status, const int32_t* __restrict__ pos0) {
  constexpr uint32_t kRowBytes = kFp8 ? kDI : 2 * kDI;  // bytes of one operand row
  constexpr int kN = G * kHI;  // MMA N: query-head rows
  constexpr int kComputeWarps = CW;
  constexpr int kComputeThreads = 32 * CW;
  constexpr int kStages = TopkCfg<CW>::kStages;
  constexpr uint32_t kKeysOff = TopkCfg<CW>::kKeysOff;
  constexpr int kQPW = G * 4 / CW > 1 ? G * 4 / CW : 1;  // queries scored per warpgroup
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages], s_dfull[kDBufs], s_dfree[kDBufs];
  __shared__ __align__(8) uint64_t s_qfull, s_qempty;
  __shared__ __align__(8) uint64_t s_drain;  // the MMA thread's last commit, before tensor memory is freed
  __shared__ float s_w[G][kHI];
  constexpr int kSelWG = CW / 4;  // selecting warpgroups: one query each at a time
  __shared__ uint32_t s_kmin[G], s_kmax[G];  // order keys: each query's visible score range
  __shared__ int s_scan[kSelWG][4];
  __shared__ int s_cnt[kSelWG][2][4];
  __shared__ int s_bin[kSelWG], s_binneed[kSelWG], s_bincnt[kSelWG], s_ncand[kSelWG];
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int vstride = (max_vis + 3) & ~3;
  // scores (float, -0 stored as +0) of query q at [q * vstride, ...), then the selection regions
  float* sScore = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)) + kKeysOff);
  uint32_t* sSel = reinterpret_cast<uint32_t*>(sScore + (size_t)G * vstride);
  const uint32_t bar_full = smem_u32(&s_full[0]), bar_empty = smem_u32(&s_empty[0]);
  const uint32_t bar_dfull = smem_u32(&s_dfull[0]), bar_dfree = smem_u32(&s_dfree[0]);
  const uint32_t bar_qfull = smem_u32(&s_qfull), bar_qempty = smem_u32(&s_qempty);

  if (warp == kComputeWarps + 1) {
    tc::tmem_alloc(smem_u32(&s_tmem), 32 * kDBufs);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int i = 0; i < kDBufs; ++i) {
      mbar_init(bar_dfull + 8 * i, 1);
      mbar_init(bar_dfree + 8 * i, kComputeWarps);
    }
    mbar_init(bar_qfull, 1);
    mbar_init(bar_qempty, 1);
    mbar_init(smem_u32(&s_drain), 1);
    fence_mbar_init();
    s_abort = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int total = total_qblocks(cu, B, G);

  if (warp == kComputeWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_map(&map_qi);
      tma_prefetch_map(&map_ki);
      uint32_t it = 0, nblk = 0;
      for (int k = blockIdx.x; k < total && !*(volatile int*)&s_abort; k += gridDim.x) {
        QBlock bk;
        if (!qblock_of(cu, cu_cmp, B, r, G, topk, max_vis, total, k, bk, pos0) || bk.ntiles == 0) continue;
        if (!mbar_wait_bounded(bar_qempty, (nblk & 1u) ^ 1u, status)) { s_abort = 1; break; }
        ++nblk;
        mbar_arrive_expect_tx(bar_qfull, kN * kRowBytes);
        tma_load_2d(base + kQIOff, &map_qi, 0, (bk.seq0 + bk.q0) * kHI, bar_qfull);
        for (int i = 0; i < bk.ntiles; ++i, ++it) {
          const uint32_t s = it % kStages;
          if (!mbar_wait_bounded(bar_empty + 8 * s, ((it / kStages) & 1u) ^ 1u, status)) { s_abort = 1; break; }
          mbar_arrive_expect_tx(bar_full + 8 * s, kTK * kRowBytes);
          tma_load_2d(base + kStageOff + s * kTileBytes, &map_ki, 0, bk.cmp0 + i * kTK, bar_full + 8 * s);
        }
      }
    }
  } else if (warp == kComputeWarps + 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t kId = kFp8 ? tc::idesc_e4m3(kTK, kN) : tc::idesc_bf16(kTK, kN, 0, 0);
      uint32_t it = 0, nblk = 0;
      for (int k = blockIdx.x; k < total && !*(volatile int*)&s_abort; k += gridDim.x) {
        QBlock bk;
        if (!qblock_of(cu, cu_cmp, B, r, G, topk, max_vis, total, k, bk, pos0) || bk.ntiles == 0) continue;
        if (!mbar_wait_bounded(bar_qfull, nblk & 1u, status)) { s_abort = 1; break; }
        ++nblk;
        for (int i = 0; i < bk.ntiles; ++i, ++it) {
          const uint32_t s = it % kStages, d = it % kDBufs;
          if (!mbar_wait_bounded(bar_full + 8 * s, (it / kStages) & 1u, status) ||
              !mbar_wait_bounded(bar_dfree + 8 * d, ((it / kDBufs) & 1u) ^ 1u, status)) {
            s_abort = 1;
            break;
          }
          tc::fence_after_sync();
          const uint32_t st = base + kStageOff + s * kTileBytes;
          if constexpr (kFp8) {
#pragma unroll
            for (int kq = 0; kq < kDI / 32; ++kq) {   // 32 one-byte elements (32 bytes) per K step
              const uint64_t a = tc::smem_desc_sw64(st + kq * 32, 512);
              const uint64_t bq = tc::smem_desc_sw64(base + kQIOff + kq * 32, 512);
              tc::mma_e4m3(tmem + d * 32, a, bq, kId, kq > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kq = 0; kq < kDI / 16; ++kq) {   // 16 bf16 elements (32 bytes) per K step
              const uint64_t a = tc::smem_desc_sw128(st + kq * 32, 16, 1024);
              const uint64_t bq = tc::smem_desc_sw128(base + kQIOff + kq * 32, 16, 1024);
              tc::mma_bf16(tmem + d * 32, a, bq, kId, kq > 0 ? 1u : 0u);
            }
          }
          tc::mma_commit(bar_dfull + 8 * d);
          tc::mma_commit(bar_empty + 8 * s);
        }
        tc::mma_commit(bar_qempty);
      }
      // every MMA this thread issued has completed before tensor memory is freed (also after an abort)
      tc::mma_commit(smem_u32(&s_drain));
      mbar_wait_bounded(smem_u32(&s_drain), 0, status);
    }
  } else {
    // ---------------- compute warps: scores, then selection ----------------
    const int g = warp >> 2, quad = warp & 3;  // warpgroup g scores queries kQPW g ... of the block
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int rowl = quad * 32 + lane;
    uint32_t it = 0;
    for (int k = blockIdx.x; k < total; k += gridDim.x) {
      QBlock bk;
      if (!qblock_of(cu, cu_cmp, B, r, G, topk, max_vis, total, k, bk, pos0)) continue;
      if (tid == 0 && (bk.q0 + bk.nq + bk.p0) / r > max_vis) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
      TK_T0(tk_sc);
      if (bk.score) {
        if (tid < G * kHI) {
          const int q = tid / kHI, h = tid % kHI;
          const int64_t wr = (int64_t)(bk.seq0 + bk.q0 + q) * kHI + h;
          float wv = q < bk.nq ? __bfloat162float(w[wr]) : 0.f;
          if constexpr (kFp8) wv = q < bk.nq ? wv * __ldg(qs + wr) : 0.f;
          s_w[q][h] = wv;
        }
        if (tid < G) {
          s_kmin[tid] = 0xFFFFFFFFu;
          s_kmax[tid] = 0u;
        }
        named_sync(1, kComputeThreads);
        const bool active = g * kQPW < G;  // this warpgroup's queries exist in the tile
        // the range of each of its queries' visible scores (order keys), for the selection's buckets
        uint32_t kmn[kQPW], kmx[kQPW];
        int nvq[kQPW];
        float wq[kQPW][kHI];  // this warpgroup's head weights, in registers for the whole block
#pragma unroll
        for (int qq = 0; qq < kQPW; ++qq) {
          const int q = g * kQPW + qq;
          kmn[qq] = 0xFFFFFFFFu;
          kmx[qq] = 0u;
          nvq[qq] = q < bk.nq ? min((bk.q0 + q + bk.p0 + 1) / r, max_vis) : 0;
#pragma unroll
          for (int h = 0; h < kHI; ++h) wq[qq][h] = q < G ? s_w[q][h] : 0.f;
        }
        for (int i = 0; i < bk.ntiles; ++i, ++it) {
          const uint32_t d = it % kDBufs;
          if (!mbar_wait_bounded(bar_dfull + 8 * d, (it / kDBufs) & 1u, status)) { s_abort = 1; break; }
          tc::fence_after_sync();
          uint32_t rv[8 * kQPW];
          if (active) {
            if constexpr (kQPW == 2) tc::tmem_ld16_sync(tmem + lane_off + d * 32 + g * kQPW * kHI, rv);
            else tc::tmem_ld8_sync(tmem + lane_off + d * 32 + g * kQPW * kHI, rv);
          }
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dfree + 8 * d);
          const int j = i * kTK + rowl;
          float kscale = 1.f;
          if constexpr (kFp8) kscale = (active && j < bk.nvis_max) ? __ldg(ks + bk.cmp0 + j) : 0.f;
          if (active && j < bk.nvis_max) {
#pragma unroll
            for (int qq = 0; qq < kQPW; ++qq) {
              const int q = g * kQPW + qq;
              float sc = 0.f;
#pragma unroll
              for (int h = 0; h < kHI; ++h) sc = fmaf(wq[qq][h], fmaxf(__uint_as_float(rv[qq * kHI + h]), 0.f), sc);
              if constexpr (kFp8) sc *= kscale;
              if (sc == 0.f) sc = 0.f;  // -0 and +0 are the same score
              sScore[(size_t)q * vstride + j] = sc;
              if (j < nvq[qq]) {
                const uint32_t key = order_key(sc);
                kmn[qq] = min(kmn[qq], key);
                kmx[qq] = max(kmx[qq], key);
              }
            }
          }
        }
        if (active) {
#pragma unroll
          for (int qq = 0; qq < kQPW; ++qq) {
            const uint32_t lo = __reduce_min_sync(0xffffffffu, kmn[qq]);
            const uint32_t hi = __reduce_max_sync(0xffffffffu, kmx[qq]);
            if (lane == 0 && nvq[qq] > 0) {
              atomicMin(&s_kmin[g * kQPW + qq], lo);
              atomicMax(&s_kmax[g * kQPW + qq], hi);
            }
          }
        }
        named_sync(1, kComputeThreads);
        if (*(volatile int*)&s_abort) break;
      }
      TK_ADD(5, tk_sc);
      // ---- selection: warpgroup sg selects queries sg, sg + kSelWG, ... one at a time ----
      {
        const int sg = warp >> 2, sw = warp & 3, st = tid & 127;
        const int wg_bar = 2 + sg;
        uint32_t* hist = sSel + sg * (kSelBytes / 4);
        uint2* cand = reinterpret_cast<uint2*>(hist);
        // The bin of this warpgroup's histogram of nb bins holding the need-th largest
        // entry (thread st sums nb / 128 bins counted from the top): s_bin, the entries
        // still needed inside it (s_binneed) and its count (s_bincnt).
        auto find_bin = [&](int nb, int need) {
          const int bpt = nb / 128;
          const int hi_bin = nb - 1 - st * bpt;
          int local = 0;
          for (int kb = 0; kb < bpt; ++kb) local += (int)hist[hi_bin - kb];
          int incl = local;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
          }
          if (lane == 31) s_scan[sg][sw] = incl;
          named_sync(wg_bar, 128);
          int cum = incl - local;
          for (int ww = 0; ww < sw; ++ww) cum += s_scan[sg][ww];
          if (cum < need && need <= cum + local) {
            for (int kb = 0; kb < bpt; ++kb) {
              const int bin = hi_bin - kb;
              const int hc = (int)hist[bin];
              if (need <= cum + hc) {
                s_bin[sg] = bin;
                s_binneed[sg] = need - cum;
                s_bincnt[sg] = hc;
                break;
              }
              cum += hc;
            }
          }
          named_sync(wg_bar, 128);
        };
        for (int q = sg; q < bk.nq; q += kSelWG) {
          const int t = bk.q0 + q;
          const int64_t orow = (int64_t)(bk.seq0 + t) * k_pad;
          const int n = min((t + bk.p0 + 1) / r, max_vis);
          const int m = min(topk, n);
          const float* sc = sScore + (size_t)q * vstride;
          const bool all = n <= topk;
          // warp sw of the warpgroup owns entries [j_lo, j_hi) (seg a multiple of 128)
          const int seg = ((n + 4 * 128 - 1) / (4 * 128)) * 128;
          const int j_lo = sw * seg, j_hi = min(n, j_lo + seg);
          // selected: score > thr, then the first need_eq entries (by index) with score == thr;
          // s_cnt[sg][0 / 1][w]: the entries of warp w's segment above / equal to thr
          float thr = 0.f;
          int need_eq = 0;
          // selected entries of the earlier warps' segments: above thr / equal to it
          int gt_before = 0, eq_before = 0;
          bool from_cnt = true;  // from s_cnt (else already counted)
          int eq_total = 0;      // entries equal to thr over the whole query
          if (all) {
            if (lane == 0) {
              s_cnt[sg][0][sw] = max(0, j_hi - j_lo);
              s_cnt[sg][1][sw] = 0;
            }
            named_sync(wg_bar, 128);
          } else if (s_kmax[q] == s_kmin[q]) {
            // every visible score equal: the first m by index
            thr = key_float(s_kmax[q]);
            need_eq = m;
            if (lane == 0) {
              s_cnt[sg][0][sw] = 0;
              s_cnt[sg][1][sw] = max(0, j_hi - j_lo);
            }
            named_sync(wg_bar, 128);
          } else {
            // value-linear buckets over [vmin, vmax]: monotone in the score, so every entry of
            // a bucket above the threshold's is selected and only that bucket needs the exact order
            const float vmin = key_float(s_kmin[q]), vmax = key_float(s_kmax[q]);
            const float span = vmax - vmin;
            const float bscale = span < INFINITY ? (float)(kSelBins - 1) / span : 0.f;
            auto bucket = [&](float v) { return min((int)((v - vmin) * bscale), kSelBins - 1); };
            for (int b = st; b < kSelBins; b += 128) hist[b] = 0u;
            if (st == 0) s_ncand[sg] = 0;
            named_sync(wg_bar, 128);
            for (int j0 = 4 * st; j0 < n; j0 += 512) {
              const float4 v4 = *reinterpret_cast<const float4*>(sc + j0);
              const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (j0 + e < n) atomicAdd(&hist[bucket(vv[e])], 1u);
            }
            named_sync(wg_bar, 128);
            find_bin(kSelBins, m);
            const int b0 = s_bin[sg], need = s_binneed[sg], c = s_bincnt[sg];
            if (c <= kCand) {
              // above bucket b0: selected; bucket b0: to the candidate list.  Lane l takes
              // entries jb + 4 l .. jb + 4 l + 3 of each 128 (one 16-byte read)
              int gt0 = 0;
              for (int jb = j_lo; jb < j_hi; jb += 128) {
                const int j0 = jb + 4 * lane;
                const float4 v4 = j0 < j_hi ? *reinterpret_cast<const float4*>(sc + j0) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
                int bb[4], nc = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  bb[e] = j0 + e < j_hi ? bucket(vv[e]) : -1;
                  gt0 += bb[e] > b0 ? 1 : 0;
                  nc += bb[e] == b0 ? 1 : 0;
                }
                if (__any_sync(0xffffffffu, nc > 0)) {
                  int incl = nc;
#pragma unroll
                  for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                  }
                  int slot = 0;
                  if (lane == 31) slot = atomicAdd(&s_ncand[sg], incl);
                  slot = __shfl_sync(0xffffffffu, slot, 31) + incl - nc;
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    if (bb[e] == b0) {
                      if (slot < kCand) cand[slot] = make_uint2(order_key(vv[e]), (uint32_t)(j0 + e));
                      ++slot;
                    }
                }
              }
              gt0 = __reduce_add_sync(0xffffffffu, gt0);
              if (lane == 0) s_cnt[sg][0][sw] = gt0;
              named_sync(wg_bar, 128);
              // every warp resolves the threshold itself (no second barrier)
              uint32_t tk;
              int gc[4], ec[4];
              resolve_candidates(cand, c, need, seg, lane, tk, need_eq, gc, ec);
              thr = key_float(tk);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                if (u < sw) {
                  gt_before += s_cnt[sg][0][u] + gc[u];
                  eq_before += ec[u];
                }
                eq_total += ec[u];
              }
              from_cnt = false;
            } else {
              // more entries share the threshold bucket than the list holds (heavy ties):
              // exact radix select over the order keys, 8 bits a round
              uint32_t prefix = 0u, pmask = 0u;
              int needf = m;
              for (int round = 0; round < 4; ++round) {
                const int shift = 24 - 8 * round;
                for (int b = st; b < 256; b += 128) hist[b] = 0u;
                named_sync(wg_bar, 128);
                for (int j0 = 4 * st; j0 < n; j0 += 512) {
                  const float4 v4 = *reinterpret_cast<const float4*>(sc + j0);
                  const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const uint32_t k = order_key(vv[e]);
                    if (j0 + e < n && (k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1u);
                  }
                }
                named_sync(wg_bar, 128);
                find_bin(256, needf);
                prefix |= (uint32_t)s_bin[sg] << shift;
                pmask |= 0xFFu << shift;
                needf = s_binneed[sg];
              }
              thr = key_float(prefix);
              need_eq = needf;
              int gt = 0, eq = 0;
              for (int j = j_lo + lane; j < j_hi; j += 32) {
                const float v = sc[j];
                gt += v > thr ? 1 : 0;
                eq += v == thr ? 1 : 0;
              }
              gt = __reduce_add_sync(0xffffffffu, gt);
              eq = __reduce_add_sync(0xffffffffu, eq);
              if (lane == 0) {
                s_cnt[sg][0][sw] = gt;
                s_cnt[sg][1][sw] = eq;
              }
              named_sync(wg_bar, 128);
            }
          }
          if (from_cnt)
            for (int ww = 0; ww < 4; ++ww) {
              if (ww < sw) {
                gt_before += s_cnt[sg][0][ww];
                eq_before += s_cnt[sg][1][ww];
              }
              eq_total += s_cnt[sg][1][ww];
            }
          if (all || eq_total == need_eq) {
            // every entry equal to thr is selected: the selected set is score >= thr (all: every
            // entry).  Entry jb + 32 e + lane per round: one ballot places a round's entries in
            // index order, in consecutive slots (coalesced stores)
            const uint32_t lt = (1u << lane) - 1u;
            int at = gt_before + eq_before;
            for (int jb = j_lo; jb < j_hi; jb += 128) {
              float vv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = jb + 32 * e + lane;
                vv[e] = (!all && j < j_hi) ? sc[j] : 0.f;
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = jb + 32 * e + lane;
                const bool f = j < j_hi && (all || vv[e] >= thr);
                const uint32_t bm = __ballot_sync(0xffffffffu, f);
                if (f) idx[orow + at + __popc(bm & lt)] = bk.cmp0 + j;
                at += __popc(bm);
              }
            }
          } else {
            // write pass: lane l takes entries jb + 4 l .. jb + 4 l + 3 of each 128 (one 16-byte
            // read); a warp scan of the per-lane counts places the selected entries in index order
            for (int jb = j_lo; jb < j_hi; jb += 128) {
              const int j0 = jb + 4 * lane;
              float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
              if (!all && j0 < j_hi) v4 = *reinterpret_cast<const float4*>(sc + j0);
              const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
              bool fg[4], fe[4];
              int ng = 0, ne = 0;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const bool in = j0 + e < j_hi;
                fg[e] = in && (all || vv[e] > thr);
                fe[e] = in && !all && vv[e] == thr;
                ng += fg[e] ? 1 : 0;
                ne += fe[e] ? 1 : 0;
              }
              int ig = ng, ie = ne;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, ig, o);
                const int b = __shfl_up_sync(0xffffffffu, ie, o);
                if (lane >= o) {
                  ig += a;
                  ie += b;
                }
              }
              int pg = gt_before + ig - ng, pe = eq_before + ie - ne;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (fg[e]) idx[orow + pg + min(pe, need_eq)] = bk.cmp0 + j0 + e;
                if (fe[e] && pe < need_eq) idx[orow + pg + pe] = bk.cmp0 + j0 + e;
                pg += fg[e] ? 1 : 0;
                pe += fe[e] ? 1 : 0;
              }
              gt_before += __shfl_sync(0xffffffffu, ig, 31);
              eq_before += __shfl_sync(0xffffffffu, ie, 31);
            }
          }
          for (int i = m + st; i < k_pad; i += 128) idx[orow + i] = -1;
          named_sync(wg_bar, 128);  // s_cnt and the histogram are reused by this warpgroup's next query
        }
      }
      named_sync(1, kComputeThreads);  // every query of the block is written: its scores may be overwritten
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kComputeWarps + 1) tc::tmem_dealloc(tmem, 32 * kDBufs);
}

#ifdef CSA_TOPK_PROFILE
extern "C" int csa_topk_profile(unsigned long long* out16) {
  if (cudaMemcpyFromSymbol(out16, g_topk_prof, sizeof(unsigned long long) * 16) != cudaSuccess) return -1;
  static const unsigned long long zeros[16] = {};
  return cudaMemcpyToSymbol(g_topk_prof, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#endif

// Shared memory a CTA may use for scores: per-SM capacity split over the CTAs
// resident on it, less static arrays (under 2 KB), the 1 KB every block
// reserves, alignment slack, the fixed front part and the selection regions.
template <int CW>
static size_t topk_key_budget() {
  const size_t per_cta = 233472 / TopkCfg<CW>::kCtasPerSm;
  return per_cta - 2 * 1024 - 1024 - 1024 - TopkCfg<CW>::kKeysOff - (size_t)(CW / 4) * kSelBytes;
}

struct TopkShape {
  int G, CW;  // queries per block, compute warps (0: unsupported)
};

static TopkShape topk_tc_shape(int max_vis) {
  const size_t per_query = (size_t)((max_vis + 3) & ~3) * 4;
  if (4 * per_query <= topk_key_budget<8>()) return {4, 8};
  if (4 * per_query <= topk_key_budget<16>()) return {4, 16};
  if (2 * per_query <= topk_key_budget<8>()) return {2, 8};
  if (2 * per_query <= topk_key_budget<16>()) return {2, 16};
  return {0, 0};
}

bool indexer_topk_tc_supported(int H_I, int d_I, int max_vis, bool fp32) {
  return !fp32 && H_I == kHI && d_I == kDI && topk_tc_shape(max_vis).G > 0;
}

template <int G, int CW, bool kFp8>
static cudaError_t launch_topk_tc_t(const void* qI, const float* qs, const void* w, const void* kI, const float* ks,
                                    const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap, int max_vis, int r,
                                    int topk, int k_pad, int32_t* idx, int* status, cudaStream_t stream,
                                    const int32_t* pos0, int cmp_rows) {
  CUtensorMap mqi, mki;
  const int rows_c = cmp_rows > T_cap / r ? cmp_rows : T_cap / r;  // rows of the compressed array
  const uint64_t n_cmp_rows = (uint64_t)(rows_c > 0 ? rows_c : 1);
  if (kFp8) {
    if (!make_tmap_u8_sw64(&mqi, qI, (uint64_t)T_cap * kHI, kDI, G * kHI) ||
        !make_tmap_u8_sw64(&mki, kI, n_cmp_rows, kDI, kTK))
      return cudaErrorInvalidValue;
  } else if (!make_tmap_bf16_sw128(&mqi, qI, (uint64_t)T_cap * kHI, kDI, G * kHI) ||
             !make_tmap_bf16_sw128(&mki, kI, n_cmp_rows, kDI, kTK)) {
    return cudaErrorInvalidValue;
  }
  const size_t smem =
      1024 + TopkCfg<CW>::kKeysOff + (size_t)G * ((max_vis + 3) & ~3) * 4 + (size_t)(CW / 4) * kSelBytes;
  auto kern = indexer_topk_tc_kernel<G, CW, kFp8>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int blocks = T_cap / G + B + 1;
  const int slots = sms * TopkCfg<CW>::kCtasPerSm;
  const int grid = blocks < slots ? blocks : slots;
  kern<<<grid, TopkCfg<CW>::kThreads, smem, stream>>>(mqi, mki, static_cast<const __nv_bfloat16*>(w), qs, ks, cu,
                                                      cu_cmp, B, r, topk, k_pad, max_vis, idx, status, pos0);
  return cudaGetLastError();
}

template <bool kFp8>
static cudaError_t launch_topk_tc_any(const void* qI, const float* qs, const void* w, const void* kI, const float* ks,
                                      const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap, int max_vis, int r,
                                      int topk, int k_pad, int32_t* idx, int* status, cudaStream_t stream,
                                      const int32_t* pos0, int cmp_rows) {
  if (T_cap <= 0) return cudaSuccess;
  const TopkShape sh = topk_tc_shape(max_vis);
  if (sh.G == 4 && sh.CW == 8)
    return launch_topk_tc_t<4, 8, kFp8>(qI, qs, w, kI, ks, cu, cu_cmp, B, T_cap, max_vis, r, topk, k_pad, idx, status,
                                        stream, pos0, cmp_rows);
  if (sh.G == 2 && sh.CW == 8)
    return launch_topk_tc_t<2, 8, kFp8>(qI, qs, w, kI, ks, cu, cu_cmp, B, T_cap, max_vis, r, topk, k_pad, idx, status,
                                        stream, pos0, cmp_rows);
  if (sh.G == 4)
    return launch_topk_tc_t<4, 16, kFp8>(qI, qs, w, kI, ks, cu, cu_cmp, B, T_cap, max_vis, r, topk, k_pad, idx,
                                         status, stream, pos0, cmp_rows);
  return launch_topk_tc_t<2, 16, kFp8>(qI, qs, w, kI, ks, cu, cu_cmp, B, T_cap, max_vis, r, topk, k_pad, idx, status,
                                       stream, pos0, cmp_rows);
}

cudaError_t launch_indexer_topk_tc(const void* qI, const void* w, const void* kI, const int32_t* cu,
                                   const int32_t* cu_cmp, int B, int T_cap, int max_vis, int r, int topk, int k_pad,
                                   int32_t* idx, int* status, cudaStream_t stream, const int32_t* pos0,
                                   int cmp_rows) {
  return launch_topk_tc_any<false>(qI, nullptr, w, kI, nullptr, cu, cu_cmp, B, T_cap, max_vis, r, topk, k_pad, idx,
                                   status, stream, pos0, cmp_rows);
}

cudaError_t launch_indexer_topk_fp8(const uint8_t* qI, const float* qs, const void* w, const uint8_t* kI,
                                    const float* ks, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap,
                                    int max_vis, int r, int topk, int k_pad, int32_t* idx, int* status,
                                    cudaStream_t stream, const int32_t* pos0, int cmp_rows) {
  return launch_topk_tc_any<true>(qI, qs, w, kI, ks, cu, cu_cmp, B, T_cap, max_vis, r, topk, k_pad, idx, status,
                                  stream, pos0, cmp_rows);
}

}  // namespace csa
