// indexer_kl_tc.cu -- the dense-teacher indexer KL loss on tcgen05 tensor
// cores with TMA-fed tiles (64 heads x 128 dims, indexer 8 x 64, bf16).
//
// "DeepSeek-V4 Attention Training Systems": §3 (L_I = sum_t KL(Softmax(a_{t,C_t})
// || Softmax(i_{t,C_t})) with C_t the full visible compressed history in the
// dense-loss phase), §2 phase table (the sparse warm-up's teacher is ~O(L^2/4)
// score work), §8.2 (dense teacher scores recomputed for the loss), §9 (FP32
// loss math).
//
// In the dense phase C_t is every visible entry, a prefix of the sequence's
// compressed rows, so consecutive queries share their keys: one CTA takes a
// block of 4 queries (4 x 64 = 256 query-head rows) and streams the key prefix
// through shared memory with TMA tiled loads (128 keys x 128 dims, 128-byte
// swizzle), each tile feeding 256 rows of tensor-core work.
//   pass 1  S = Q K^T   (two M=128 tiles of query-head rows, N=128 keys, two
//           tensor-memory buffers so the next tile's MMAs run during this
//           tile's arithmetic): each row's log-sum-exp -> lse_h. Two warpgroup
//           pairs take alternate tiles (one buffer each), a thread a whole row
//           of its tile; each pair keeps a partial (reference, sum) per row,
//           merged at the end.
//   pass 2  S^T = K Q^T (M=128 keys, N=256 query-heads) and the indexer tile
//           I^T = kI qI^T (M=128 keys, N=32 = 4 queries x 8 heads): one thread
//           per (key, query) forms p(j) = mean_h exp(s_h - lse_h), the indexer
//           logit i = sum_h w_h ReLU(.), and accumulates sum p ln p, sum p i
//           and the student's log-sum-exp;  KL = sum p ln p - sum p i + lse_i.
// Warp roles: warps 0-15 compute (four warpgroups, one tensor-memory lane per
// thread; four warps per scheduler hide the exp2 and FMA latencies), warp 16
// issues the TMA loads, warp 17 allocates tensor memory and issues the MMAs.
// Pass 2 threads copy each score tile to registers and release it at once;
// pass 1 threads release theirs once both 64-column chunks are loaded.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "kl_blocks.cuh"
#include "tma.cuh"

namespace csa {

#ifdef CSA_KL_PROFILE
// Profiling build only: cycles per (role, site), summed over warps.
__device__ unsigned long long g_kl_prof[48];
#define KL_T0(v) const long long v = clock64()
#define KL_ADD(site, v) \
  do {                  \
    if (lane == 0) s_prof[warp][site] += (unsigned long long)(clock64() - (v)); \
  } while (0)
#define KL_CNT(site) \
  do {               \
    if (lane == 0) s_prof[warp][site] += 1ull; \
  } while (0)
#else
#define KL_T0(v)
#define KL_ADD(site, v)
#define KL_CNT(site)
#endif

namespace {

constexpr int kQB = 4;          // queries per block
constexpr int kNH = 64;         // heads
constexpr int kDim = 128;       // head dim
constexpr int kHI = 8;          // indexer heads
constexpr int kDI = 64;         // indexer head dim
constexpr int kTK = 128;        // keys per tile
constexpr int kStages = 3;
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kThreads = kComputeThreads + 64;

constexpr uint32_t kQRegion = kQB * kNH * 128;       // 32 KB: 256 rows x 64 dims
constexpr uint32_t kQOff = 0;
constexpr uint32_t kQIOff = 2 * kQRegion;            // 4 KB: 32 rows x 64 dims
constexpr uint32_t kKRegion = kTK * 128;             // 16 KB
constexpr uint32_t kStageK = 2 * kKRegion;           // 32 KB
constexpr uint32_t kStageBytes = kStageK + kKRegion; // + kI tile (16 KB)
constexpr uint32_t kStageOff = kQIOff + 4096;        // 1024-aligned
constexpr uint32_t kSmemBytes = kStageOff + kStages * kStageBytes;
static_assert(kStageOff % 1024 == 0, "stage alignment");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBufCols = 256;  // pass 1 score buffer d at columns [256 d, 256 d + 256)
constexpr uint32_t kColI = 256;     // indexer tile columns in pass 2 (inside buffer 1)

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

using klb::Block;

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
indexer_kl_dense_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                           const __grid_constant__ CUtensorMap map_qi, const __grid_constant__ CUtensorMap map_ki,
                           const __nv_bfloat16* __restrict__ w, const int32_t* __restrict__ cu,
                           const int32_t* __restrict__ cu_cmp, int B, int r, float scale_log2,
                           float* __restrict__ kl_rows, int32_t* __restrict__ csize, int* status,
                           float* __restrict__ teacher_lse, float* __restrict__ student_lse,
                           const int32_t* __restrict__ pos0) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
  __shared__ __align__(8) uint64_t s_sfull[2], s_sfree[2], s_qfull, s_qempty;
  __shared__ __align__(8) uint64_t s_drain;  // the MMA thread's last commit, before tensor memory is freed
  __shared__ __align__(16) float s_L[kQB][kNH];  // per (query, head) minus the log2 normaliser over C_t
  __shared__ float s_w[kQB][kHI];
  __shared__ float s_red[kComputeWarps][4];  // per compute warp: A, B, mI, lI
  __shared__ float s_ml[2][kQB * kNH][2];    // pass 1 per column half: row max, row sum
  __shared__ int s_abort;
#ifdef CSA_KL_PROFILE
  __shared__ unsigned long long s_prof[kThreads / 32][16];
#endif

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#ifdef CSA_KL_PROFILE
  if (lane == 0)
    for (int i = 0; i < 16; ++i) s_prof[warp][i] = 0;
#endif
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = smem_u32(&s_full[0]), bar_empty = smem_u32(&s_empty[0]);
  const uint32_t bar_sfull = smem_u32(&s_sfull[0]), bar_sfree = smem_u32(&s_sfree[0]);
  const uint32_t bar_qfull = smem_u32(&s_qfull), bar_qempty = smem_u32(&s_qempty);

  if (warp == kComputeWarps + 1) {
    tc::tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(bar_sfull + 8 * d, 1);
      mbar_init(bar_sfree + 8 * d, kComputeWarps);  // one arrival per compute warp
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
  const int total = klb::total_blocks<kQB>(cu, B);

  if (warp == kComputeWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_qi);
      tma_prefetch_map(&map_ki);
      uint32_t it = 0, nblk = 0;
      for (int k = blockIdx.x; k < total && !*(volatile int*)&s_abort; k += gridDim.x) {
        Block bk;
        if (!klb::block_of<kQB, kTK>(cu, cu_cmp, B, r, total, k, bk, pos0) || bk.ntiles == 0) continue;
        if (!mbar_wait_bounded(bar_qempty, (nblk & 1u) ^ 1u, status)) { s_abort = 1; break; }
        ++nblk;
        mbar_arrive_expect_tx(bar_qfull, 2 * kQRegion + kQB * kHI * 128);
        for (int rg = 0; rg < 2; ++rg)
          for (int m = 0; m < 2; ++m)
            tma_load_2d(base + kQOff + rg * kQRegion + m * 16384, &map_q, rg * 64, (bk.seq0 + bk.q0) * kNH + m * 128,
                        bar_qfull);
        tma_load_2d(base + kQIOff, &map_qi, 0, (bk.seq0 + bk.q0) * kHI, bar_qfull);
        for (int pass = 0; pass < 2; ++pass) {
          for (int i = 0; i < bk.ntiles; ++i, ++it) {
            const uint32_t s = it % kStages;
            KL_T0(t_e);
            if (!mbar_wait_bounded(bar_empty + 8 * s, ((it / kStages) & 1u) ^ 1u, status)) { s_abort = 1; break; }
            KL_ADD(0, t_e);
            KL_CNT(1);
            const uint32_t st = base + kStageOff + s * kStageBytes;
            mbar_arrive_expect_tx(bar_full + 8 * s, pass == 0 ? kStageK : kStageBytes);
            tma_load_2d(st, &map_k, 0, bk.cmp0 + i * kTK, bar_full + 8 * s);
            tma_load_2d(st + kKRegion, &map_k, 64, bk.cmp0 + i * kTK, bar_full + 8 * s);
            if (pass == 1) tma_load_2d(st + kStageK, &map_ki, 0, bk.cmp0 + i * kTK, bar_full + 8 * s);
          }
          if (s_abort) break;
        }
      }
    }
  } else if (warp == kComputeWarps + 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t kIdP1 = tc::idesc_bf16(128, kTK, 0, 0);
      constexpr uint32_t kIdP2 = tc::idesc_bf16(kTK, kQB * kNH, 0, 0);
      constexpr uint32_t kIdI = tc::idesc_bf16(kTK, kQB * kHI, 0, 0);
      uint32_t it = 0, nblk = 0, nf0 = 0, nf1 = 0;
      for (int k = blockIdx.x; k < total && !*(volatile int*)&s_abort; k += gridDim.x) {
        Block bk;
        if (!klb::block_of<kQB, kTK>(cu, cu_cmp, B, r, total, k, bk, pos0) || bk.ntiles == 0) continue;
        if (!mbar_wait_bounded(bar_qfull, nblk & 1u, status)) { s_abort = 1; break; }
        ++nblk;
        for (int pass = 0; pass < 2; ++pass) {
          for (int i = 0; i < bk.ntiles; ++i, ++it) {
            const uint32_t s = it % kStages;
            // pass 1 alternates the two score buffers (even tiles of a block: buffer 0, so every
            // row's partial sums take the same tiles whatever the block's place in the grid);
            // a pass 2 tile takes both
            const uint32_t d = (uint32_t)i & 1u;
            const bool use0 = pass == 1 || d == 0, use1 = pass == 1 || d == 1;
            KL_T0(m_f);
            const bool okf = mbar_wait_bounded(bar_full + 8 * s, (it / kStages) & 1u, status);
            KL_ADD(0, m_f);
            KL_T0(m_s);
            if (!okf || (use0 && !mbar_wait_bounded(bar_sfree, (nf0 & 1u) ^ 1u, status)) ||
                (use1 && !mbar_wait_bounded(bar_sfree + 8, (nf1 & 1u) ^ 1u, status))) {
              s_abort = 1;
              break;
            }
            KL_ADD(1, m_s);
            KL_CNT(2);
            tc::fence_after_sync();
            const uint32_t st = base + kStageOff + s * kStageBytes;
            if (pass == 0) {
#pragma unroll
              for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int ks = 0; ks < kDim / 16; ++ks) {
                  const uint64_t a = tc::smem_desc_sw128(base + kQOff + (ks >> 2) * kQRegion + g * 16384 + (ks & 3) * 32,
                                                         16, 1024);
                  const uint64_t bd = tc::smem_desc_sw128(st + (ks >> 2) * kKRegion + (ks & 3) * 32, 16, 1024);
                  tc::mma_bf16(tmem + d * kBufCols + g * kTK, a, bd, kIdP1, ks > 0 ? 1u : 0u);
                }
            } else {
#pragma unroll
              for (int ks = 0; ks < kDim / 16; ++ks) {
                const uint64_t a = tc::smem_desc_sw128(st + (ks >> 2) * kKRegion + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = tc::smem_desc_sw128(base + kQOff + (ks >> 2) * kQRegion + (ks & 3) * 32, 16, 1024);
                tc::mma_bf16(tmem, a, bd, kIdP2, ks > 0 ? 1u : 0u);
              }
#pragma unroll
              for (int ks = 0; ks < kDI / 16; ++ks) {
                const uint64_t a = tc::smem_desc_sw128(st + kStageK + ks * 32, 16, 1024);
                const uint64_t bd = tc::smem_desc_sw128(base + kQIOff + ks * 32, 16, 1024);
                tc::mma_bf16(tmem + kColI, a, bd, kIdI, ks > 0 ? 1u : 0u);
              }
            }
            if (use0) { tc::mma_commit(bar_sfull); ++nf0; }
            if (use1) { tc::mma_commit(bar_sfull + 8); ++nf1; }
            tc::mma_commit(bar_empty + 8 * s);
          }
          if (s_abort) break;
        }
        tc::mma_commit(bar_qempty);  // Q / qI free once this block's MMAs are done
      }
      // every MMA this thread issued has completed before tensor memory is freed (also after an abort)
      tc::mma_commit(smem_u32(&s_drain));
      mbar_wait_bounded(smem_u32(&s_drain), 0, status);
    }
  } else {
    // ---------------- compute warpgroups ----------------
    const int wg = warp >> 2;                // warpgroup 0..3
    const int quad = warp & 3;               // tensor-memory lane quadrant
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int rowl = quad * 32 + lane;       // tensor-memory lane of this thread
    uint32_t nf0 = 0, nf1 = 0;               // score-buffer uses, as counted by the MMA warp
    for (int k = blockIdx.x; k < total; k += gridDim.x) {
      Block bk;
      if (!klb::block_of<kQB, kTK>(cu, cu_cmp, B, r, total, k, bk, pos0)) continue;
      if (bk.ntiles == 0) {
        if (tid < bk.nq) {
          kl_rows[bk.seq0 + bk.q0 + tid] = 0.f;
          csize[bk.seq0 + bk.q0 + tid] = 0;
        }
        continue;
      }
      if (tid < kQB * kHI) {
        const int q = tid / kHI, h = tid % kHI;
        s_w[q][h] = q < bk.nq ? __bfloat162float(w[(int64_t)(bk.seq0 + bk.q0 + q) * kHI + h]) : 0.f;
      }
      // ---- pass 1: row (query, head) online log-sum-exp ----
      // Warpgroup pair wg >> 1 takes the tiles of score buffer wg >> 1 (every other tile): whole
      // 128-column rows of M-tile wg & 1, in two 64-column chunks, so the two pairs work on
      // consecutive tiles at once rather than all sixteen warps waiting on one.
      {
        const int mt = wg & 1;
        const int half = wg >> 1;  // the pair: its buffer, and the slot of its partial (m, l) of the row
        const int q = 2 * mt + (rowl >> 6), h = rowl & 63;
        const int nvis = (bk.q0 + q + bk.p0 + 1) / r;
        float m = -INFINITY, l = 0.f;
        for (int i = 0; i < bk.ntiles; ++i) {
          const uint32_t d = (uint32_t)i & 1u;
          if (d != (uint32_t)half) {  // the other pair's tile
            if (d) ++nf1; else ++nf0;
            continue;
          }
          KL_T0(c_w1);
          if (!mbar_wait_bounded(bar_sfull + 8 * d, (d ? nf1 : nf0) & 1u, status)) { s_abort = 1; break; }
          KL_ADD(0, c_w1);
          KL_T0(c_l1);
          tc::fence_after_sync();
          float x[kTK / 2];
          auto load = [&](int col) {
            uint32_t rs[kTK / 2];
            tc::tmem_ld64_sync(tmem + lane_off + d * kBufCols + mt * kTK + col, rs);
#pragma unroll
            for (int jj = 0; jj < kTK / 2; ++jj) x[jj] = __uint_as_float(rs[jj]);
          };
          auto release = [&]() {
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {  // the barrier counts an arrival from each of the sixteen compute warps
              mbar_arrive(bar_sfree + 8 * d);
              mbar_arrive(bar_sfree + 8 * d);
            }
            if (d) ++nf1; else ++nf0;
          };
          // the 64 columns in x, of which the first nv are visible, folded into (m, l)
          auto fold = [&](int nv) {
            if (nv < kTK / 2) {  // only the last tile of a row is partial
#pragma unroll
              for (int c = 0; c < kTK / 2; ++c) x[c] = c < nv ? x[c] : -INFINITY;
            }
            // sum over the chunk of 2^(x scale - ref): packed pairs, one f32x2 FMA and one f32x2
            // add per two columns
            auto chunk_sum = [&](float ref) {
              const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nr2 = f2_pack(-ref, -ref);
              uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
              for (int c = 0; c < kTK / 2; c += 4) {
                float a0, a1, a2, a3;
                f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), sc2, nr2), a0, a1);
                f2_unpack(f2_fma(f2_pack(x[c + 2], x[c + 3]), sc2, nr2), a2, a3);
                acc0 = f2_add(acc0, f2_pack(ex2(a0), ex2(a1)));
                acc1 = f2_add(acc1, f2_pack(ex2(a2), ex2(a3)));
              }
              float s0, s1, s2, s3;
              f2_unpack(acc0, s0, s1);
              f2_unpack(acc1, s2, s3);
              return (s0 + s1) + (s2 + s3);
            };
            // After the row's first chunk, its running reference m stays put: every term is taken
            // against it, with no chunk maximum, which holds while no score exceeds m by 64 or more
            // (each term below 2^64, the sum far from the float range's end). A chunk whose sum
            // reaches 2^64 (or overflows) is redone against its own maximum, as the first is.
            bool exact = m == -INFINITY;
            if (!exact) {
              const float ts = chunk_sum(m);
              if (ts < 1.8446744e19f) l += ts;  // 2^64; false for inf and NaN
              else exact = true;
            }
            if (exact) {
              float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
              for (int c = 0; c < kTK / 2; c += 4) {
                t0 = max3f(t0, x[c], x[c + 1]);
                t1 = max3f(t1, x[c + 2], x[c + 3]);
              }
              const float mn = fmaxf(m, fmaxf(t0, t1) * scale_log2);  // scale > 0: max commutes with it
              if (mn != -INFINITY) {
                const float ts = chunk_sum(mn);
                l = l * ex2(m - mn) + ts;
                m = mn;
              }
            }
          };
          load(0);
          KL_ADD(1, c_l1);
          KL_T0(c_c1);
          fold(nvis - i * kTK);
          load(kTK / 2);  // the buffer is released once both chunks are in registers
          release();
          fold(nvis - i * kTK - kTK / 2);
          KL_ADD(2, c_c1);
          KL_CNT(7);
        }
        KL_T0(c_m);
        s_ml[half][mt * kTK + rowl][0] = m;
        s_ml[half][mt * kTK + rowl][1] = l;
        named_sync(1, kComputeThreads);
        if (half == 0 && q < kQB) {  // merge the row's two partials
          const float m2 = s_ml[1][mt * kTK + rowl][0], l2 = s_ml[1][mt * kTK + rowl][1];
          const float mx = fmaxf(m, m2);
          const float ls = (mx == -INFINITY) ? 0.f : l * ex2(m - mx) + l2 * ex2(m2 - mx);
          s_L[q][h] = (ls > 0.f) ? -(mx + __log2f(ls)) : -INFINITY;  // negated; -inf: contributes nothing
          if (teacher_lse != nullptr && q < bk.nq)  // natural units, for the indexer backward
            teacher_lse[(int64_t)(bk.seq0 + bk.q0 + q) * kNH + h] =
                (ls > 0.f) ? (mx + __log2f(ls)) * 0.6931471805599453f : -INFINITY;
        }
        KL_ADD(9, c_m);
      }
      named_sync(1, kComputeThreads);
      if (*(volatile int*)&s_abort) break;  // uniform: read after the barrier
      // ---- pass 2: one thread per key, warpgroup q = query q ----
      const int q = wg;
      const int nvis_q = (bk.q0 + q + bk.p0 + 1) / r;
      const bool q_ok = q < bk.nq;
      float A = 0.f, Bs = 0.f, mI = -INFINITY, lI = 0.f;
      for (int i = 0; i < bk.ntiles; ++i) {
        KL_T0(c_w2);
        if (!mbar_wait_bounded(bar_sfull, nf0 & 1u, status) || !mbar_wait_bounded(bar_sfull + 8, nf1 & 1u, status)) {
          s_abort = 1;
          break;
        }
        KL_ADD(3, c_w2);
        KL_T0(c_l2);
        tc::fence_after_sync();
        float x[kNH];
        uint32_t ri[8];
        {
          uint32_t rs[kNH];
          tc::tmem_ld64_ld8_sync(tmem + lane_off + q * kNH, tmem + lane_off + kColI + q * kHI, rs, ri);
#pragma unroll
          for (int jj = 0; jj < kNH; ++jj) x[jj] = __uint_as_float(rs[jj]);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_sfree);
          mbar_arrive(bar_sfree + 8);
        }
        ++nf0;
        ++nf1;
        KL_ADD(4, c_l2);
        KL_T0(c_c2);
        const int j = i * kTK + rowl;  // entry index within the sequence
        if (q_ok && j < nvis_q) {
          const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
          uint64_t pa = f2_pack(0.f, 0.f), pb = pa;
          const float4* L4 = reinterpret_cast<const float4*>(&s_L[q][0]);  // -lse_h
#pragma unroll
          for (int h4 = 0; h4 < kNH / 4; ++h4) {
            const float4 L = L4[h4];
            float a0, a1, a2, a3;
            f2_unpack(f2_fma(f2_pack(x[4 * h4 + 0], x[4 * h4 + 1]), sc2, f2_pack(L.x, L.y)), a0, a1);
            f2_unpack(f2_fma(f2_pack(x[4 * h4 + 2], x[4 * h4 + 3]), sc2, f2_pack(L.z, L.w)), a2, a3);
            pa = f2_add(pa, f2_pack(ex2(a0), ex2(a1)));
            pb = f2_add(pb, f2_pack(ex2(a2), ex2(a3)));
          }
          float p0, p1, p2, p3;
          f2_unpack(pa, p0, p1);
          f2_unpack(pb, p2, p3);
          const float p = ((p0 + p1) + (p2 + p3)) * (1.f / kNH);
          float iv = 0.f;
#pragma unroll
          for (int hh = 0; hh < kHI; ++hh) iv = fmaf(s_w[q][hh], fmaxf(__uint_as_float(ri[hh]), 0.f), iv);
          if (p > 0.f) A = fmaf(p, __logf(p), A);
          Bs = fmaf(p, iv, Bs);
          // the student's sum against a held reference: the thread's first key sets it, and a
          // key whose term reaches 2^64 against it moves it
          const float e = __expf(iv - mI);
          if (e < 1.8446744e19f) {
            lI += e;  // not taken while mI == -inf (e = inf)
          } else {
            lI = lI * __expf(mI - iv) + 1.f;
            mI = iv;
          }
        }
        KL_ADD(5, c_c2);
        KL_CNT(8);
      }
      KL_T0(c_end);
      // reduce the per-key partials over the warpgroup's 128 threads
      {
        float a = A, bs = Bs, mm = mI, ll = lI;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          a += __shfl_xor_sync(0xffffffffu, a, o);
          bs += __shfl_xor_sync(0xffffffffu, bs, o);
          const float m2 = __shfl_xor_sync(0xffffffffu, mm, o);
          const float l2 = __shfl_xor_sync(0xffffffffu, ll, o);
          const float mx = fmaxf(mm, m2);
          ll = (mx == -INFINITY) ? 0.f : ll * __expf(mm - mx) + l2 * __expf(m2 - mx);
          mm = mx;
        }
        if (lane == 0) {
          s_red[warp][0] = a;
          s_red[warp][1] = bs;
          s_red[warp][2] = mm;
          s_red[warp][3] = ll;
        }
      }
      named_sync(1, kComputeThreads);
      if (tid < kQB && tid < bk.nq) {
        const int qq = tid;
        float a = 0.f, bs = 0.f, mm = -INFINITY;
        for (int ww = 0; ww < 4; ++ww) {
          a += s_red[qq * 4 + ww][0];
          bs += s_red[qq * 4 + ww][1];
          mm = fmaxf(mm, s_red[qq * 4 + ww][2]);
        }
        float ll = 0.f;
        for (int ww = 0; ww < 4; ++ww) {
          const float m2 = s_red[qq * 4 + ww][2];
          if (m2 != -INFINITY) ll += s_red[qq * 4 + ww][3] * __expf(m2 - mm);
        }
        const int nvis = (bk.q0 + qq + bk.p0 + 1) / r;
        kl_rows[bk.seq0 + bk.q0 + qq] = nvis > 0 ? a - bs + (mm + __logf(ll)) : 0.f;
        if (student_lse != nullptr) student_lse[bk.seq0 + bk.q0 + qq] = nvis > 0 ? mm + __logf(ll) : -INFINITY;
        csize[bk.seq0 + bk.q0 + qq] = nvis;
      }
      named_sync(1, kComputeThreads);
      KL_ADD(6, c_end);
      if (*(volatile int*)&s_abort) break;
    }
  }
#ifdef CSA_KL_PROFILE
  if (lane == 0) {
    const int role = warp < kComputeWarps ? 0 : (warp == kComputeWarps + 1 ? 1 : 2);
    for (int i = 0; i < 16; ++i) atomicAdd(&g_kl_prof[role * 16 + i], s_prof[warp][i]);
  }
#endif

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kComputeWarps + 1) tc::tmem_dealloc(tmem, kTmemCols);
}

#ifdef CSA_KL_PROFILE
extern "C" int csa_kl_profile(unsigned long long* out48) {
  if (cudaMemcpyFromSymbol(out48, g_kl_prof, sizeof(unsigned long long) * 48) != cudaSuccess) return -1;
  static const unsigned long long zeros[48] = {};
  return cudaMemcpyToSymbol(g_kl_prof, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#endif

bool indexer_kl_dense_tc_supported(const KLArgs& a, bool fp32) {
  return !fp32 && a.idx == nullptr && a.H == kNH && a.d == kDim && a.H_I == kHI && a.d_I == kDI;
}

__global__ void kl_zero_rows_kernel(float* __restrict__ kl_rows, int32_t* __restrict__ csize, int T_cap,
                                    float* __restrict__ teacher_lse, int H, float* __restrict__ student_lse) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T_cap; i += gridDim.x * blockDim.x) {
    kl_rows[i] = 0.f;
    csize[i] = 0;
    if (student_lse) student_lse[i] = -INFINITY;  // rows without a C_t keep -inf
  }
  if (teacher_lse)
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < (int64_t)T_cap * H;
         i += (int64_t)gridDim.x * blockDim.x)
      teacher_lse[i] = -INFINITY;
}

cudaError_t launch_kl_zero_rows(float* kl_rows, int32_t* csize, int T_cap, float* teacher_lse, int H,
                                float* student_lse, cudaStream_t stream) {
  kl_zero_rows_kernel<<<152, 256, 0, stream>>>(kl_rows, csize, T_cap, teacher_lse, H, student_lse);
  return cudaGetLastError();
}

cudaError_t launch_indexer_kl_dense_tc(const KLArgs& a, cudaStream_t stream) {
  if (a.T_cap <= 0) return cudaSuccess;
  CUtensorMap mq, mk, mqi, mki;
  // the compressed arrays hold at most T_cap / r rows
  const int rows_c = a.cmp_rows > a.T_cap / a.r ? a.cmp_rows : a.T_cap / a.r;
  const uint64_t n_cmp_rows = (uint64_t)(rows_c > 0 ? rows_c : 1);
  if (!make_tmap_bf16_sw128(&mq, a.q, (uint64_t)a.T_cap * kNH, kDim, 128) ||
      !make_tmap_bf16_sw128(&mk, a.k_cmp, n_cmp_rows, kDim, kTK) ||
      !make_tmap_bf16_sw128(&mqi, a.qI, (uint64_t)a.T_cap * kHI, kDI, kQB * kHI) ||
      !make_tmap_bf16_sw128(&mki, a.kI, n_cmp_rows, kDI, kTK))
    return cudaErrorInvalidValue;
  kl_zero_rows_kernel<<<152, 256, 0, stream>>>(a.kl_rows, a.csize, a.T_cap, a.teacher_lse, a.H, a.student_lse);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t smem = kSmemBytes + 1024;
  auto kern = indexer_kl_dense_tc_kernel;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int blocks = (a.T_cap + kQB - 1) / kQB + a.B;  // upper bound on query blocks
  const int grid = blocks < sms ? blocks : sms;
  constexpr float kLog2e = 1.4426950408889634f;
  kern<<<grid, kThreads, smem, stream>>>(
      mq, mk, mqi, mki, static_cast<const __nv_bfloat16*>(a.w), a.cu, a.cu_cmp, a.B, a.r, a.scale * kLog2e,
      a.kl_rows, a.csize, a.status, a.teacher_lse, a.student_lse, a.pos0);
  return cudaGetLastError();
}

}  // namespace csa
