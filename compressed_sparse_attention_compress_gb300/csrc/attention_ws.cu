// attention_ws.cu -- warp-specialised selected / HCA / window attention forward
// on tcgen05 tensor cores, 64 heads x 128 dims, one shared K = V head.
//
// "DeepSeek-V4 Attention Training Systems": §2 phase table (top-k compressed
// entries + local window; HCA reads every completed ratio-128 entry plus the
// window), §8.2 (selected MQA attention over a flat global index list returning
// output and LSE; compressed ids combined with window ids), §9 (FP32 sink,
// FP32 softmax).
//
// Tiles are transposed as in the two-CTA kernel: the 128 gathered keys are the
// M dimension, the 64 heads the N dimension.
//   S^T[key, h]  = K[key, :] . Q[h, :]        (M=128, N=64, K=128 dims)
//   O^T[dim, h] += V^T[dim, key] P^T[key, h]  (M=128, N=64, K=128 keys)
// An N=64 MMA reads 6 KB of shared-memory operands per 48 cycles, so a tile
// needs about 770 tensor cycles; the kernel is organised to keep that pipe fed.
//
// One CTA per SM runs two independent query streams (groups).  Each group has
// its own two-stage key-tile ring, its own Q buffer, P^T buffer and tensor-
// memory columns (S^T 64 + O^T 64 + running sums 64), so neither waits on the
// other:
//   a producer warp per group: resolve each tile's rows (index list read
//     one tile ahead), skip compressed tiles with no valid entry, gather rows
//     with 16-byte cp.async copies that arrive on the stage's mbarrier;
//   softmax warps (8 per group): thread (key, head half) reads 32 head scores
//     of its key, keeps the per-head running reference lazily (a block vote
//     rescales only when a score exceeds it by 2^8), writes its half of the
//     key's bf16 P^T row, and at the end of a query reduces the per-thread
//     sums and writes O / LSE;
//   an MMA warp per group: issues QK of the next tile as soon as S^T has been
//     read and the tile gathered, then PV of the current tile once its P^T is
//     written (shared-memory descriptors precomputed, waits that sleep).
// Precision: the weights enter P^T as bf16 (relative error up to 2^-9), and
// every normaliser (the output's, lse, lse_cmp) is the sum of those rounded
// weights, so the output is a convex combination of the value rows with the
// weights the tensor cores used.  The running reference is the exact maximum
// while a query has seen fewer than kExactKeys keys: one key can then carry
// most of the weight, and at the exact maximum its weight is exactly 1.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "ws_sync.cuh"

namespace csa {

#ifdef CSA_WS_PROFILE
// Profiling build only: cycles per (role, site), summed over warps.
__device__ unsigned long long g_ws_prof[48];
#define WS_T0(v) const long long v = clock64()
#define WS_ADD(site, v) \
  do {                  \
    if (lane == 0) s_prof[warp][site] += (unsigned long long)(clock64() - (v)); \
  } while (0)
#define WS_CNT(site) \
  do {               \
    if (lane == 0) s_prof[warp][site] += 1ull; \
  } while (0)
#else
#define WS_T0(v)
#define WS_ADD(site, v)
#define WS_CNT(site)
#endif

namespace {

using namespace ws;

constexpr int kTK = 128, kNH = 64, kDim = 128;
constexpr int kSoftWarps = 8;                              // per group
constexpr int kProdWarps = 1;                              // per group
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kProdWarp0 = 2 * kSoftWarps;                 // warps 16, 17
constexpr int kMmaWarp = kProdWarp0 + 2 * kProdWarps;      // warps 18, 19: one MMA issuer per group
constexpr int kRowsPerProd = kTK / kProdThreads;           // 4
constexpr int kThreads = 32 * (kMmaWarp + 2);
constexpr float kTau = 8.f;                                // lazy-max slack, log2 units
constexpr int kExactKeys = 32;                             // exact maximum until this many keys were seen

constexpr uint32_t kQRegion = kNH * 128;                   // 8 KB: 64 rows x 64 dims
constexpr uint32_t kQBytes = 2 * kQRegion;                 // 16 KB per group
constexpr uint32_t kTileRegion = kTK * 128;                // 16 KB
constexpr uint32_t kTileBytes = 2 * kTileRegion;           // 32 KB
constexpr uint32_t kQOff = 0;
constexpr uint32_t kStageOff = 2 * kQBytes;                // [group][stage]
constexpr uint32_t kPOff = kStageOff + 4 * kTileBytes;     // [group]
constexpr uint32_t kSmem = kPOff + 2 * kTK * 128;          // 192 KB

enum : int { kFirst = 1, kLast = 2, kWinStart = 4, kDone = 8, kCmp = 16 };

struct Meta {
  int row;
  int flags;
  int nvalid;  // keys of the tile that take part
};

__device__ __forceinline__ int ord_of(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float float_of(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF); }

// Sum 32 per-thread values over a warp and return, in lane l, the sum of entry l
// (five halving exchange steps: a lane keeps the half its lane bit selects).
__device__ __forceinline__ float warp_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int half = 16 >> step;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < half) {
        const float send = upper ? v[j] : v[j + half];
        const float keep = upper ? v[j + half] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
  return v[0];
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
attention_ws_kernel(int kind, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cmp,
                    const __nv_bfloat16* __restrict__ k_raw, const int32_t* __restrict__ idx, int k_pad,
                    const float* __restrict__ sink, const int32_t* __restrict__ cu,
                    const int32_t* __restrict__ cu_cmp, int B, int T_cap, int r, int window, float scale_log2,
                    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, float* __restrict__ lse_cmp,
                    int* status,
                    const int32_t* __restrict__ pos0) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_full[2][2], s_empty[2][2];
  __shared__ __align__(8) uint64_t s_drain[2];  // each MMA thread's last commit, before tensor memory is freed
  __shared__ __align__(8) uint64_t s_qfull[2], s_qempty[2], s_sfull[2], s_sfree[2], s_pfull[2], s_odone[2],
      s_ofree[2];
  __shared__ Meta s_meta[2][2];
  __shared__ int s_rows[2][2][kTK];
  __shared__ __align__(16) float s_m[2][kNH];
  __shared__ __align__(16) float s_nm[2][kNH];  // -s_m
  __shared__ float s_alpha[2][kNH], s_dm[2][kNH], s_inv[2][kNH];
  __shared__ int s_wmax[2][4][kNH];
  __shared__ float s_lsum[2][4][kNH];
  __shared__ int s_abort;
#ifdef CSA_WS_PROFILE
  __shared__ unsigned long long s_prof[kThreads / 32][16];
#endif

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#ifdef CSA_WS_PROFILE
  if (lane == 0)
    for (int i = 0; i < 16; ++i) s_prof[warp][i] = 0;
#endif
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  auto full_bar = [&](int g, int s) { return smem_u32(&s_full[g][s]); };
  auto empty_bar = [&](int g, int s) { return smem_u32(&s_empty[g][s]); };

  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_u32(&s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int g = 0; g < 2; ++g) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(full_bar(g, s), 2 * kProdThreads);  // cp.async arrivals + per-warp release
        mbar_init(empty_bar(g, s), 1);
      }
      mbar_init(smem_u32(&s_qfull[g]), 2 * kProdThreads);
      mbar_init(smem_u32(&s_qempty[g]), 1);
      mbar_init(smem_u32(&s_sfull[g]), 1);
      mbar_init(smem_u32(&s_sfree[g]), kSoftWarps);
      mbar_init(smem_u32(&s_pfull[g]), kSoftWarps);
      mbar_init(smem_u32(&s_odone[g]), 1);
      mbar_init(smem_u32(&s_ofree[g]), kSoftWarps);
    }
    mbar_init(smem_u32(&s_drain[0]), 1);
    mbar_init(smem_u32(&s_drain[1]), 1);
    fence_mbar_init();
    s_abort = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  const int cmp_limit = kind == kAttnWindow ? 0 : __ldg(cu_cmp + B);
  const int raw_limit = __ldg(cu + B);

  if (warp >= kProdWarp0 && warp < kMmaWarp) {
    // =================== producers: group g, lane pt owns rows pt + 32 i of every tile ===================
    const int g = warp - kProdWarp0;
    const int pt = lane;
    const uint32_t qb = base + kQOff + g * kQBytes;
    uint32_t n = 0, nq = 0;  // tiles and queries produced
    bool alive = true;
    for (int ord = g; alive; ord += 2) {
      const int qi = blockIdx.x + ord * gridDim.x;
      if (qi >= T_cap) break;
      const int row = T_cap - 1 - qi;  // latest rows (most keys) first
      const int b = owner_sequence(cu, B, row);
      if (b < 0) continue;             // capacity rows are written by another kernel
      const int seq0 = __ldg(cu + b);
      const int t = row - seq0;
      const int p0 = pos0 ? __ldg(pos0 + b) : 0;  // position of the sequence's first row here
      const int nvis = (kind == kAttnWindow || r <= 0) ? 0 : (t + p0 + 1) / r;
      const int cmp0 = kind == kAttnWindow ? 0 : __ldg(cu_cmp + b);
      const int w0 = max(0, t - window + 1);
      const int nwin = t - w0 + 1;
      const int ncs = kind == kAttnCSA ? k_pad : (kind == kAttnHCA ? nvis : 0);
      const int nct = (ncs + kTK - 1) / kTK;
      const int ntl = nct + (nwin + kTK - 1) / kTK;
      int pre[kRowsPerProd];
#pragma unroll
      for (int i = 0; i < kRowsPerProd; ++i) pre[i] = -1;
      auto prefetch = [&](int it) {
        if (kind == kAttnCSA && it < nct) {
          const int32_t* src = idx + (int64_t)row * k_pad;
#pragma unroll
          for (int i = 0; i < kRowsPerProd; ++i) {
            const int slot = it * kTK + pt + 32 * i;
            pre[i] = slot < k_pad ? __ldg(src + slot) : -1;
          }
        }
      };
      auto resolve = [&](int it, int key, int pv) -> int {
        int rr = -1;
        if (it < nct) {
          if (kind == kAttnCSA) {
            if (pv >= 0) {
              if (pv < cmp0 || pv >= cmp0 + nvis || pv >= cmp_limit) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
              else rr = pv;
            }
          } else if (it * kTK + key < nvis) {
            rr = cmp0 + it * kTK + key;
          }
        } else {
          const int wi = (it - nct) * kTK + key;
          if (wi < nwin && seq0 + w0 + wi < raw_limit) rr = seq0 + w0 + wi;
        }
        return rr;
      };
      prefetch(0);
      bool first = true;
      for (int it = 0; it < ntl; ++it) {
        WS_T0(p_res);
        int rr[kRowsPerProd];
        bool any = false;
#pragma unroll
        for (int i = 0; i < kRowsPerProd; ++i) {
          rr[i] = resolve(it, pt + 32 * i, pre[i]);
          any = any || rr[i] >= 0;
        }
        prefetch(it + 1);
        if (it < nct && !__any_sync(0xffffffffu, any)) continue;  // empty compressed tile
        WS_ADD(2, p_res);
        const uint32_t st = n & 1u;
        WS_T0(p_empty);
        bool ok = mbar_wait_bounded(empty_bar(g, st), ((n >> 1) & 1u) ^ 1u, status);
        WS_ADD(0, p_empty);
        WS_T0(p_q);
        if (first && nq > 0) ok = ok && mbar_wait_bounded(smem_u32(&s_qempty[g]), (nq - 1) & 1u, status);
        WS_ADD(1, p_q);
        WS_T0(p_gather);
        if (__any_sync(0xffffffffu, !ok || *abort_flag != 0)) {
          *abort_flag = 1;
          alive = false;
          break;
        }
        if (first) {  // this query's Q (64 heads x 128 dims, swizzled K-major)
#pragma unroll 4
          for (int i = pt; i < kNH * 16; i += kProdThreads) {
            const int h = i >> 4, c = i & 15;
            cp_async_16(qb + (c >> 3) * kQRegion + tc::sw128_offset(h, c & 7),
                        q + ((int64_t)row * kNH + h) * kDim + c * 8);
          }
          arrive_cp_async(smem_u32(&s_qfull[g]));
          __syncwarp();
          if (lane == 0) arrive_warp(smem_u32(&s_qfull[g]));
          ++nq;
        }
        const bool cmpt = it < nct;
        const __nv_bfloat16* ks = cmpt ? k_cmp : k_raw;
        int nval = 0;
#pragma unroll
        for (int i = 0; i < kRowsPerProd; ++i) nval += __popc(__ballot_sync(0xffffffffu, rr[i] >= 0));
        const uint32_t kb = base + kStageOff + (g * 2 + st) * kTileBytes;
#pragma unroll
        for (int i = 0; i < kRowsPerProd; ++i) s_rows[g][st][pt + 32 * i] = rr[i];
        // coalesced gather: eight lanes per 256-byte row, four rows per step;
        // lane chunk c (16 bytes) of dims [8c, 8c+8) and its partner chunk c + 8
        const int c = lane & 7, sub = lane >> 3;
#pragma unroll
        for (int j = 0; j < kTK / 4; ++j) {
          const int key = 4 * j + sub;
          const int rk = __shfl_sync(0xffffffffu, rr[j / 8], 4 * (j % 8) + sub);
          const __nv_bfloat16* src = ks + (int64_t)(rk < 0 ? 0 : rk) * kDim + c * 8;
          const uint32_t dst = kb + tc::sw128_offset(key, c);
          cp_async_16_zfill(dst, src, rk >= 0);
          cp_async_16_zfill(dst + kTileRegion, src + 64, rk >= 0);
        }
        if (pt == 0) {
          const int flags = (first ? kFirst : 0) | (cmpt ? kCmp : 0) | (it == nct ? kWinStart : 0) |
                            (it == ntl - 1 ? kLast : 0);
          s_meta[g][st] = Meta{row, flags, nval};
        }
        arrive_cp_async(full_bar(g, st));
        __syncwarp();
        if (lane == 0) arrive_warp(full_bar(g, st));  // release: publishes s_rows / s_meta
        WS_ADD(3, p_gather);
        WS_CNT(4);
        first = false;
        ++n;
      }
    }
    if (alive) {  // end-of-stream marker for this group
      const uint32_t st = n & 1u;
      const bool ok = mbar_wait_bounded(empty_bar(g, st), ((n >> 1) & 1u) ^ 1u, status);
      if (__any_sync(0xffffffffu, !ok)) {
        *abort_flag = 1;
      } else {
        if (pt == 0) s_meta[g][st] = Meta{-1, kDone, 0};
        mbar_arrive(full_bar(g, st));
        __syncwarp();
        if (lane == 0) arrive_warp(full_bar(g, st));
      }
    }
    cp_async_wait<0>();
  } else if (warp >= kMmaWarp) {
    // =================== MMA issuer of group g: whatever is ready, PV first ===================
    const int g = warp - kMmaWarp;
    if (lane == 0) {
      constexpr uint32_t kIdQK = tc::idesc_bf16(kTK, kNH, 0, 0);
      constexpr uint32_t kIdPV = tc::idesc_bf16(kDim, kNH, 1, 1);
      // descriptors of K-step 0; a K-step adds its byte offset / 16 to the address field
      const uint64_t dq = tc::smem_desc_sw128(base + kQOff + g * kQBytes, 16, 1024);
      const uint64_t dp = tc::smem_desc_sw128(base + kPOff + g * (kTK * 128), 1024, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(base + kStageOff + (g * 2) * kTileBytes, 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(base + kStageOff + (g * 2) * kTileBytes, kTileRegion, 1024);
      constexpr uint64_t kStageStep = kTileBytes >> 4;
      const uint32_t t_s = tmem + g * 128, t_o = tmem + g * 128 + kNH;
      uint32_t kq = 0, kp = 0, nqq = 0, nqp = 0;  // QKs / PVs issued, queries started by QK / PV
      bool end = false;                           // the end-of-stream tile was seen
      uint64_t last = globaltimer_ns();
      while (!(end && kp == kq)) {
        bool progress = false;
        // PV(kp): frees the stage for the producer as early as possible
        if (kp < kq && mbar_test(smem_u32(&s_pfull[g]), kp & 1u)) {
          const uint32_t sp = kp & 1u;
          const bool first = (s_meta[g][sp].flags & kFirst) != 0;
          if (!first || nqp == 0 || mbar_test(smem_u32(&s_ofree[g]), (nqp - 1) & 1u)) {
            if (first) ++nqp;
            tc::fence_after_sync();
            const uint64_t dv = dv0 + sp * kStageStep;
#pragma unroll
            for (int ks = 0; ks < kTK / 16; ++ks) {
              const uint32_t off = (ks * 2048) >> 4;
              tc::mma_bf16(t_o, dv + off, dp + off, kIdPV, (first && ks == 0) ? 0u : 1u);
            }
            tc::mma_commit(smem_u32(&s_odone[g]));
            tc::mma_commit(empty_bar(g, sp));
            ++kp;
            progress = true;
          }
        }
        // QK(kq): its tile is gathered and the softmax has read S^T(kq - 1)
        if (!end && kq < kp + 2 && mbar_test(full_bar(g, kq & 1u), (kq >> 1) & 1u)) {
          const uint32_t st = kq & 1u;
          const int flags = s_meta[g][st].flags;
          if (flags & kDone) {
            end = true;
            progress = true;
          } else if ((kq == 0 || mbar_test(smem_u32(&s_sfree[g]), (kq - 1) & 1u)) &&
                     (!(flags & kFirst) || mbar_test(smem_u32(&s_qfull[g]), nqq & 1u))) {
            if (flags & kFirst) ++nqq;
            tc::fence_after_sync();
            const uint64_t dk = dk0 + st * kStageStep;
#pragma unroll
            for (int ks = 0; ks < kDim / 16; ++ks) {
              const uint32_t off = ((ks >> 2) * kTileRegion + (ks & 3) * 32) >> 4;
              const uint32_t offq = ((ks >> 2) * kQRegion + (ks & 3) * 32) >> 4;
              tc::mma_bf16(t_s, dk + off, dq + offq, kIdQK, ks > 0 ? 1u : 0u);
            }
            tc::mma_commit(smem_u32(&s_sfull[g]));
            if (flags & kLast) tc::mma_commit(smem_u32(&s_qempty[g]));
            ++kq;
            progress = true;
          }
        }
        if (progress) {
          WS_CNT(6);
          last = globaltimer_ns();
        } else {
          if (*abort_flag) break;
          if (globaltimer_ns() - last > kWaitLimitNs) {
            raise_status(status, CSA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          // sleep on the barrier the next issue waits for, instead of spinning on the
          // scheduler the softmax warps share: the next QK's if one is due, else the PV's
          if (!end && kq < kp + 2) {
            const uint32_t sf = smem_u32(&s_sfree[g]);
            if (kq > 0 && !mbar_test(sf, (kq - 1) & 1u)) mbar_sleep(sf, (kq - 1) & 1u, 500);
            else mbar_sleep(full_bar(g, kq & 1u), (kq >> 1) & 1u, 500);
          } else if (kp < kq) {
            mbar_sleep(smem_u32(&s_pfull[g]), kp & 1u, 500);
          } else {
            __nanosleep(64);
          }
        }
      }
      // every MMA this thread issued has completed before tensor memory is freed (also after an abort)
      tc::mma_commit(smem_u32(&s_drain[g]));
      mbar_wait_bounded(smem_u32(&s_drain[g]), 0, status);
    }
  } else {
    // =================== softmax: group g, warp sw = (head half, lane quadrant) ===================
    const int g = warp / kSoftWarps, sw = warp % kSoftWarps;
    const int quad = sw & 3, hh = sw >> 2;
    const int key = quad * 32 + lane;            // tensor-memory lane: key of the tile / head dim
    const int tig = tid - g * kSoftThreads;      // thread index within the group
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + g * 128 + hh * 32;
    const uint32_t t_o = tmem + lane_off + g * 128 + kNH + hh * 32;
    // this thread's running per-head sums of p over its key (32 heads) live in
    // tensor memory next to the accumulators, which keeps registers for the scores
    // The sums are of the bf16-rounded weights that enter P^T, so the output is a
    // convex combination of the value rows with exactly the weights the tensor
    // cores used, and the LSEs are those of the same weights.
    const uint32_t t_l = tmem + lane_off + 256 + g * kNH + hh * 32;
    const int gbar = 1 + g;
    float* m_g = s_m[g];
    const uint32_t prow = base + kPOff + g * (kTK * 128);
    uint32_t k = 0;
    int row = -1;
    bool have_o = false;
    int seen = 0;  // keys of the current query in the tiles before this one
    auto load_l = [&](float (&v)[32], uint32_t at) {
#pragma unroll
      for (int c0 = 0; c0 < 32; c0 += 16) {
        uint32_t rv[16];
        tc::tmem_ld16_sync(at + c0, rv);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(rv[j]);
      }
    };
    for (uint32_t n = 0;; ++n) {
      const uint32_t st = n & 1u;
      WS_T0(s_full_t);
      const bool okf = mbar_wait_bounded(full_bar(g, st), (n >> 1) & 1u, status);
      WS_ADD(0, s_full_t);
      if (bar_or(gbar, kSoftThreads, !okf || *abort_flag != 0)) {
        *abort_flag = 1;
        break;
      }
      const Meta mt = s_meta[g][st];
      if (mt.flags & kDone) break;
      const bool fresh = (mt.flags & kFirst) != 0;  // the running reference is not set yet
      if (fresh) {
        row = mt.row;
        have_o = false;
        seen = 0;
      }
      if ((mt.flags & kWinStart) && lse_cmp != nullptr) {  // compressed candidates done: their normaliser
        float tmp[32];
        if (fresh) {  // no compressed tile was taken: the sums are empty
#pragma unroll
          for (int j = 0; j < 32; ++j) tmp[j] = 0.f;
        } else {
          load_l(tmp, t_l);
        }
        s_lsum[g][quad][hh * 32 + lane] = warp_sum32(tmp, lane);
        bar_sync(gbar, kSoftThreads);
        if (tig < kNH) {
          const float l = s_lsum[g][0][tig] + s_lsum[g][1][tig] + s_lsum[g][2][tig] + s_lsum[g][3][tig];
          lse_cmp[(int64_t)row * kNH + tig] = l > 0.f ? (m_g[tig] + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
        bar_sync(gbar, kSoftThreads);
      }
      const bool valid = s_rows[g][st][key] >= 0;
      // ---- 32 head scores of this key ----
      WS_T0(s_sf);
      bool ok = mbar_wait_bounded(smem_u32(&s_sfull[g]), k & 1u, status);
      WS_ADD(1, s_sf);
      WS_T0(s_ex);
      tc::fence_after_sync();
      float t[32];
      {
        uint32_t rs[32];
        tc::tmem_ld32_sync(t_s, rs);
#pragma unroll
        for (int j = 0; j < 32; ++j) t[j] = __uint_as_float(rs[j]);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_sfree[g]));
      // log2 weights against the running reference: t_h = s_h * scale*log2(e) - m_h
      float excess = -INFINITY;
      if (valid) {
        if (fresh) {
#pragma unroll
          for (int j = 0; j < 32; ++j) t[j] *= scale_log2;
          excess = INFINITY;
        } else {
          const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {  // packed pairs against -m (kept negated in shared memory)
            const float4 nm4 = reinterpret_cast<const float4*>(s_nm[g] + hh * 32)[j4];
            f2_unpack(f2_fma(f2_pack(t[4 * j4 + 0], t[4 * j4 + 1]), sc2, f2_pack(nm4.x, nm4.y)), t[4 * j4 + 0],
                      t[4 * j4 + 1]);
            f2_unpack(f2_fma(f2_pack(t[4 * j4 + 2], t[4 * j4 + 3]), sc2, f2_pack(nm4.z, nm4.w)), t[4 * j4 + 2],
                      t[4 * j4 + 3]);
            excess = fmaxf(excess, fmaxf(fmaxf(t[4 * j4 + 0], t[4 * j4 + 1]), fmaxf(t[4 * j4 + 2], t[4 * j4 + 3])));
          }
        }
      }
      WS_ADD(2, s_ex);
      // the previous PV must be done before P^T / O^T are touched
      WS_T0(s_vote);
      // one vote per tile: a score above the reference by more than the slack, or a
      // failed wait (the abort is then decided uniformly inside).  The previous tile's
      // PV keeps running meanwhile: it is waited for only where P^T / O^T are touched.
      const bool bad = !ok || *abort_flag != 0;
      bool pv_done = k == 0;
      // the reference is the exact running maximum while a query has seen fewer than
      // kExactKeys keys (with few candidates one key can carry most of the weight:
      // its weight is then exactly 1 in P^T, free of bf16 rounding), and lags by up
      // to kTau after that
      const float tau = seen < kExactKeys ? 0.f : kTau;
      if (bar_or(gbar, kSoftThreads, excess > tau || bad)) {
        // new reference: the tile's per-head column maxima (t + m is the scaled score)
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float sc = t[j] + (fresh ? 0.f : m_g[hh * 32 + j]);
          const int v = __reduce_max_sync(0xffffffffu, ord_of(valid ? sc : -INFINITY));
          if (lane == 0) s_wmax[g][quad][hh * 32 + j] = v;
        }
        bool ok2 = true;
        if (!pv_done) ok2 = mbar_wait_bounded(smem_u32(&s_odone[g]), (k - 1) & 1u, status);
        pv_done = true;
        if (bar_or(gbar, kSoftThreads, bad || !ok2)) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after_sync();
        if (tig < kNH) {
          const float mo = fresh ? -INFINITY : m_g[tig];
          float mn = mo;
#pragma unroll
          for (int w = 0; w < 4; ++w) mn = fmaxf(mn, float_of(s_wmax[g][w][tig]));
          s_alpha[g][tig] = (mo == -INFINITY) ? 1.f : ex2(mo - mn);
          s_dm[g][tig] = (fresh ? 0.f : mo) - mn;
          m_g[tig] = mn;
          s_nm[g][tig] = -mn;
        }
        bar_sync(gbar, kSoftThreads);
#pragma unroll
        for (int j = 0; j < 32; ++j) t[j] += s_dm[g][hh * 32 + j];
        if (!fresh) {  // the sums follow the new reference
#pragma unroll
          for (int c0 = 0; c0 < 32; c0 += 16) {
            uint32_t rv[16];
            tc::tmem_ld16_sync(t_l + c0, rv);
#pragma unroll
            for (int j = 0; j < 16; ++j) rv[j] = __float_as_uint(__uint_as_float(rv[j]) * s_alpha[g][hh * 32 + c0 + j]);
            tc::tmem_st16(t_l + c0, rv);
          }
          tc::tmem_wait_st();
        }
        if (have_o) {  // O^T row `key` (a head dim), this warp's 32 head columns
#pragma unroll
          for (int c0 = 0; c0 < 32; c0 += 16) {
            uint32_t ro[16];
            tc::tmem_ld16_sync(t_o + c0, ro);
#pragma unroll
            for (int j = 0; j < 16; ++j) ro[j] = __float_as_uint(__uint_as_float(ro[j]) * s_alpha[g][hh * 32 + c0 + j]);
            tc::tmem_st16(t_o + c0, ro);
          }
          tc::tmem_wait_st();
        }
      }
      WS_ADD(4, s_vote);
      WS_T0(s_od);
      // P^T is overwritten below: the previous tile's PV must be done reading it
      if (!pv_done && !mbar_wait_bounded(smem_u32(&s_odone[g]), (k - 1) & 1u, status)) *abort_flag = 1;
      tc::fence_after_sync();
      WS_ADD(3, s_od);
      WS_T0(s_p);
      // ---- this thread's half of the key's P^T row: 32 heads -> 4 swizzled 16-byte chunks ----
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int h = c * 8 + 2 * j;
          pk[j] = valid ? pack_bf16x2(ex2(t[h]), ex2(t[h + 1])) : 0u;
          t[h] = bf16_lo(pk[j]);  // t now holds the weight as written
          t[h + 1] = bf16_hi(pk[j]);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + tc::sw128_offset(key, hh * 4 + c)),
                     "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]));
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_pfull[g]));
      // running sums (off the P^T -> PV path)
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t lv[16];
        if (fresh) {
#pragma unroll
          for (int j = 0; j < 16; ++j) lv[j] = __float_as_uint(t[c2 * 16 + j]);
        } else {
          tc::tmem_ld16_sync(t_l + c2 * 16, lv);
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float a, b;
            f2_unpack(f2_add(f2_pack(__uint_as_float(lv[j]), __uint_as_float(lv[j + 1])),
                             f2_pack(t[c2 * 16 + j], t[c2 * 16 + j + 1])), a, b);
            lv[j] = __float_as_uint(a);
            lv[j + 1] = __float_as_uint(b);
          }
        }
        tc::tmem_st16(t_l + c2 * 16, lv);
      }
      tc::tmem_wait_st();
      seen += mt.nvalid;
      WS_ADD(5, s_p);
      WS_CNT(7);
      have_o = true;
      ++k;
      if (mt.flags & kLast) {
        // ---- end of the query: per-head normaliser, sink, O / l, LSE ----
        WS_T0(s_epi);
        ok = mbar_wait_bounded(smem_u32(&s_odone[g]), (k - 1) & 1u, status);
        if (bar_or(gbar, kSoftThreads, !ok)) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after_sync();
        {
          float lt[32];
          load_l(lt, t_l);
          s_lsum[g][quad][hh * 32 + lane] = warp_sum32(lt, lane);
        }
        bar_sync(gbar, kSoftThreads);
        if (tig < kNH) {
          float l = s_lsum[g][0][tig] + s_lsum[g][1][tig] + s_lsum[g][2][tig] + s_lsum[g][3][tig];
          float m = m_g[tig];
          float corr = 1.f;
          if (sink != nullptr) {  // the sink enters the normaliser only (it has no value row)
            const float s2 = __ldg(sink + tig) * 1.4426950408889634f;
            const float mf = fmaxf(m, s2);
            corr = (m == -INFINITY) ? 0.f : ex2(m - mf);
            l = l * corr + ex2(s2 - mf);
            m = mf;
          }
          s_inv[g][tig] = l > 0.f ? corr / l : 0.f;
          lse[(int64_t)row * kNH + tig] = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
        bar_sync(gbar, kSoftThreads);
        {
          uint32_t ro[32];
          tc::tmem_ld32_sync(t_o, ro);
          __nv_bfloat16* orow = out + ((int64_t)row * kNH + hh * 32) * kDim + key;  // this thread's head dim
#pragma unroll
          for (int j = 0; j < 32; ++j)
            orow[(int64_t)j * kDim] = __float2bfloat16(__uint_as_float(ro[j]) * s_inv[g][hh * 32 + j]);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_ofree[g]));
        WS_ADD(6, s_epi);
      }
    }
  }
#ifdef CSA_WS_PROFILE
  if (lane == 0) {
    const int role = warp < kProdWarp0 ? 0 : (warp < kMmaWarp ? 1 : 2);
    for (int i = 0; i < 16; ++i) atomicAdd(&g_ws_prof[role * 16 + i], s_prof[warp][i]);
  }
#endif

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, 512);
}

// Capacity rows (>= cu[B]): zero output, -inf LSEs.
__global__ void attention_capacity_rows_kernel(const int32_t* __restrict__ cu, int B, int T_cap,
                                               __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                               float* __restrict__ lse_cmp) {
  const int64_t first = __ldg(cu + B);
  const int64_t n_out = ((int64_t)T_cap - first) * kNH * kDim;
  const int64_t n_lse = ((int64_t)T_cap - first) * kNH;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_out; i += (int64_t)gridDim.x * blockDim.x)
    out[first * kNH * kDim + i] = __float2bfloat16(0.f);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_lse; i += (int64_t)gridDim.x * blockDim.x) {
    lse[first * kNH + i] = -INFINITY;
    if (lse_cmp) lse_cmp[first * kNH + i] = -INFINITY;
  }
}

bool attention_ws_supported(const AttnArgs& a, bool fp32) {
  return !fp32 && a.H == kNH && a.d == kDim && a.v_cmp == nullptr && a.v_raw == nullptr;
}

cudaError_t launch_attention_ws(AttnKind kind, const AttnArgs& a, cudaStream_t stream) {
  if (a.T_cap <= 0) return cudaSuccess;
  const size_t smem = kSmem + 1024;
  cudaError_t err = cudaFuncSetAttribute(attention_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  attention_capacity_rows_kernel<<<sms, 256, 0, stream>>>(a.cu, a.B, a.T_cap, static_cast<__nv_bfloat16*>(a.out),
                                                          a.lse, a.lse_cmp);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int grid = (a.T_cap + 1) / 2 < sms ? (a.T_cap + 1) / 2 : sms;
  constexpr float kLog2e = 1.4426950408889634f;
  attention_ws_kernel<<<grid, kThreads, smem, stream>>>(
      (int)kind, static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_cmp),
      static_cast<const __nv_bfloat16*>(a.k_raw), a.idx, a.k_pad, a.sink, a.cu, a.cu_cmp, a.B, a.T_cap, a.r,
      a.window, a.scale * kLog2e, static_cast<__nv_bfloat16*>(a.out), a.lse, a.lse_cmp, a.status, a.pos0);
  return cudaGetLastError();
}

#ifdef CSA_WS_PROFILE
extern "C" int csa_ws_profile(unsigned long long* out48) {
  if (cudaMemcpyFromSymbol(out48, g_ws_prof, sizeof(unsigned long long) * 48) != cudaSuccess) return -1;
  static const unsigned long long zeros[48] = {};
  return cudaMemcpyToSymbol(g_ws_prof, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#endif

}  // namespace csa
