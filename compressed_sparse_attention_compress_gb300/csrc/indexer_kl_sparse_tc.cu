// indexer_kl_sparse_tc.cu -- the selected-set (sparse-mode) indexer KL loss on
// tcgen05 tensor cores (64 heads x 128 dims, indexer 8 x 64, bf16).
//
// "DeepSeek-V4 Attention Training Systems": §3 (L_I = sum_t KL(Softmax(a_{t,C_t})
// || Softmax(i_{t,C_t}))), §2 phase table (sparse mode: C_t is the selected
// set), §8.2 ("recompute sparse/dense teacher scores for the indexer loss"), §9
// (FP32 loss math).
//
// C_t is query t's own selected set, so no key tile is shared between queries:
// the kernel gathers each query's selected compressed rows, as the selected
// attention does, into 128-key tiles and runs two passes over them.
//   pass 1  S^T = K Q^T (M = 128 keys, N = 64 heads): per head the sum
//           Z_h = sum_j exp(s_hj - r_h) around a reference r_h (the attention's
//           lse_cmp, within a few units of the true log normaliser), so that
//           L_h = r_h + log Z_h is the teacher's exact per-head normaliser;
//   pass 2  S^T again and I^T = kI qI^T (M = 128 keys, N = 16: 8 indexer heads
//           and 8 zero rows): per key p(j) = mean_h exp(s_hj - L_h), the logit
//           i_j = sum_h w_h ReLU(.), and the sums sum p ln p, sum p i and the
//           student's log-sum-exp; KL_t = sum p ln p - sum p i + lse_i.
// Warp roles: six producer warps (warp 8 resolves each tile's index slots, all
// six gather a share of its rows with coalesced 16-byte cp.async copies: one
// warp keeps only a few copies in flight, so the gather rate grows with the
// number of issuing warps), one MMA warp (warp 14), and two compute warpgroups
// (warps 0-7) that take alternate tiles through four tensor-memory score
// buffers: thread = key of the tile, all 64 head scores of it.
// When the selected set fits in four tiles (k_pad <= 512), pass 1 gathers the
// kI rows with the keys and its S^T / I^T tiles stay in tensor memory (one
// slot per tile) for pass 2, which then neither gathers nor multiplies again;
// the next query's scores wait for both warpgroups to release the set.
// Rows with an empty C_t are written by a fill kernel beforehand (KL 0).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "ws_sync.cuh"

namespace csa {

namespace {

using namespace ws;

constexpr int kNH = 64, kDim = 128, kHI = 8, kDI = 64;
constexpr int kTK = 128;                               // keys per tile
constexpr int kStages = 3;
constexpr int kComputeWarps = 8;                       // two warpgroups
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kProdWarps = 6;                          // warps 8-13
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kProdWarp0 = kComputeWarps;
constexpr int kMmaWarp = kProdWarp0 + kProdWarps;      // warp 14 (warp 15 idles)
constexpr int kThreads = 32 * 16;
// Register split (setmaxnreg): 512 threads launch with 128 registers each; the
// two compute warpgroups take 184 and the producer / MMA warpgroups give
// theirs down to 72, which sums to the launch's 512 x 128.
constexpr uint32_t kComputeRegs = 184, kSideRegs = 72;
static_assert(256 * kComputeRegs + 256 * kSideRegs <= 512 * 128, "register split");

constexpr uint32_t kQRegion = kNH * 128;               // 8 KB: 64 heads x 64 dims
constexpr uint32_t kQBytes = 2 * kQRegion;             // 16 KB per query slot
constexpr uint32_t kQIBytes = 16 * 128;                // 2 KB: 8 indexer heads + 8 zero rows
constexpr uint32_t kAuxBytes = 512;                    // per query slot: reference (64 floats) + w (8 bf16)
constexpr uint32_t kKRegion = kTK * 128;               // 16 KB: 128 keys x 64 dims
constexpr uint32_t kStageBytes = 3 * kKRegion;         // K (two regions) + kI
constexpr uint32_t kQOff = 0;                          // [2 slots]
constexpr uint32_t kQIOff = 2 * kQBytes;               // [2 slots]
constexpr uint32_t kAuxOff = kQIOff + 2 * kQIBytes;    // [2 slots]
constexpr uint32_t kStageOff = kAuxOff + 1024;         // 37 KB, 1024-aligned
constexpr uint32_t kIdxOff = kStageOff + kStages * kStageBytes;  // [2 slots][k_pad] index rows
constexpr uint32_t kSmem = kIdxOff;                                // + 8 k_pad bytes
static_assert(kStageOff % 1024 == 0, "stage alignment");

constexpr int kBufs = 4;                               // score buffers (warpgroup d % 2 reads buffer d)
constexpr uint32_t kBufCols = 64;                      // S^T buffer d at columns 64 d
constexpr uint32_t kIdxCol = 256;                      // I^T buffer d at columns 256 + 16 d
constexpr int kMaxB = 256;                             // sequences whose offsets are kept on chip

enum : int { kFirst = 1, kLastP1 = 2, kLast = 4, kPass2 = 8, kDone = 16 };

struct TileMeta {
  int flags;
  uint32_t mask[4];  // valid keys of the tile (bit = key % 32 of word key / 32)
};

struct QueryRec {
  int row;       // packed row of the query
  int ntl;       // tiles per pass
  int nvalid;    // |C_t|
};

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

// Sum 64 per-thread values over a warp; lane l returns the sums of entries l
// and 32 + l (two transposing halving reductions).
__device__ __forceinline__ void warp_sum64_t(float (&v)[64], int lane, float& s0, float& s1) {
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    float u[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) u[j] = v[32 * part + j];
#pragma unroll
    for (int step = 0; step < 5; ++step) {
      const int o = 16 >> step;
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (j < o) {
          const float send = upper ? u[j] : u[j + o];
          const float keep = upper ? u[j + o] : u[j];
          u[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
    }
    if (part == 0) s0 = u[0]; else s1 = u[0];
  }
}

}  // namespace

// kKeep (a query's selected set fits in kBufs tiles): one gather and one S^T
// per tile; the query's S^T tiles stay in tensor memory from pass 1 to pass 2
// (slot = tile), so pass 2 reads them again instead of gathering and
// multiplying the keys a second time; the next query's scores wait for the
// compute warps to release the whole set.
template <bool kKeep>
__global__ void __launch_bounds__(kThreads, 1)
indexer_kl_sparse_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cmp,
                            const __nv_bfloat16* __restrict__ qI, const __nv_bfloat16* __restrict__ w,
                            const __nv_bfloat16* __restrict__ kI, const int32_t* __restrict__ idx, int k_pad,
                            const float* __restrict__ lse_ref, const int32_t* __restrict__ cu,
                            const int32_t* __restrict__ cu_cmp, int B, int T_cap, int r, float scale_log2,
                            float* __restrict__ kl_rows, int32_t* __restrict__ csize, int* status,
                            float* __restrict__ teacher_lse, float* __restrict__ student_lse,
                            const int32_t* __restrict__ pos0) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
  __shared__ __align__(8) uint64_t s_sfull[kBufs], s_sfree[kBufs], s_qfull[2], s_qempty[2], s_rfull[2], s_rempty[2];
  __shared__ __align__(8) uint64_t s_ifull[2];  // a query's index row landed in its slot
  __shared__ __align__(8) uint64_t s_setfree;   // kKeep: a query's score set was read by the compute warps
  __shared__ __align__(8) uint64_t s_drain;
  __shared__ TileMeta s_meta[kStages];     // written by the resolver, per stage
  __shared__ TileMeta s_bmeta[kBufs];      // copied by the MMA thread, per score buffer
  __shared__ int s_cu[kMaxB + 1], s_cc[kMaxB + 1], s_p0[kMaxB];  // the packing, on chip
  __shared__ QueryRec s_qrec[2];
  __shared__ int s_rows[kStages][kTK];
  __shared__ __align__(16) float s_ref[kNH];  // reference r_h, log2 units (negated)
  __shared__ __align__(16) float s_nL[kNH];   // -L_h, log2 units
  __shared__ float s_w[kHI];
  __shared__ float s_z[kComputeWarps][kNH];
  __shared__ float s_red[kComputeWarps][4];
  __shared__ int s_bad;                       // a reference too far below the scores
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = smem_u32(&s_full[0]), bar_empty = smem_u32(&s_empty[0]);
  const uint32_t bar_sfull = smem_u32(&s_sfull[0]), bar_sfree = smem_u32(&s_sfree[0]);
  const uint32_t bar_qfull = smem_u32(&s_qfull[0]), bar_qempty = smem_u32(&s_qempty[0]);
  const uint32_t bar_rfull = smem_u32(&s_rfull[0]), bar_rempty = smem_u32(&s_rempty[0]);

  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_u32(&s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 2 * kProdThreads);  // per producer warp: 32 cp.async arrivals + a release of 32
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(bar_sfull + 8 * i, 2);       // the MMA commit + the MMA thread's release of s_bmeta
      mbar_init(bar_sfree + 8 * i, 4);       // the four warps of the warpgroup that reads the buffer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_qfull + 8 * i, 2 * kProdThreads);  // Q, qI, reference and w copies of the producer warps
      mbar_init(bar_qempty + 8 * i, 2);      // the MMA commit after the query + the compute warps' read
      mbar_init(bar_rfull + 8 * i, 1);
      mbar_init(bar_rempty + 8 * i, kComputeWarps);
      mbar_init(smem_u32(&s_ifull[i]), 2 * kProdThreads);  // the producer warps' copies
    }
    mbar_init(smem_u32(&s_drain), 1);
    mbar_init(smem_u32(&s_setfree), kComputeWarps);
    fence_mbar_init();
    s_abort = 0;
    s_bad = 0;
  }
  // the zero rows of both qI slots (the MMA's N = 16 pads the 8 indexer heads)
  for (int i = tid; i < 2 * 8 * 8; i += kThreads) {
    const int slot = i >> 6, row = 8 + ((i >> 3) & 7), c = i & 7;
    *reinterpret_cast<uint4*>(smem_raw + (base - smem_u32(smem_raw)) + kQIOff + slot * kQIBytes +
                              tc::sw128_offset(row, c)) = make_uint4(0u, 0u, 0u, 0u);
  }
  for (int i = tid; i <= B; i += kThreads) {
    s_cu[i] = __ldg(cu + i);
    s_cc[i] = __ldg(cu_cmp + i);
    if (i < B) s_p0[i] = pos0 ? __ldg(pos0 + i) : 0;
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  // sequence owning packed row `row`: the largest b with cu[b] <= row < cu[b + 1], or -1
  auto seq_of = [&](int row) -> int {
    if (B <= 0 || row < 0 || row >= s_cu[B]) return -1;
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_cu[mid] <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  volatile int* abort_flag = &s_abort;
  const int cmp_limit = s_cc[B];

  if (warp >= kProdWarp0 && warp < kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kSideRegs));
    // ============ producers: warp 8 resolves the slots, both gather 64 rows each ============
    const int pw = warp - kProdWarp0;
    const bool resolver = pw == 0;
    uint32_t n = 0, nq = 0;  // tiles and (non-empty) queries produced
    bool alive = true;
    // the next query of this CTA at or after ord (capacity rows skipped), or -1
    auto next_query = [&](int ord) -> int {
      for (;; ++ord) {
        const int qi = blockIdx.x + ord * gridDim.x;
        if (qi >= T_cap) return -1;
        if (seq_of(T_cap - 1 - qi) >= 0) return ord;
      }
    };
    // copy a query's index row into slot `slot` (both warps, 16-byte chunks)
    uint8_t* smem_gen = smem_raw + (base - smem_u32(smem_raw));
    auto fetch_idx = [&](int ord, int slot) {
      const int row = T_cap - 1 - (blockIdx.x + ord * gridDim.x);
      const int32_t* src = idx + (int64_t)row * k_pad;
      const uint32_t dst = base + kIdxOff + (uint32_t)slot * k_pad * 4u;
      for (int c = pw * 32 + lane; c < k_pad / 4; c += kProdThreads) cp_async_16(dst + 16u * c, src + 4 * c);
      arrive_cp_async(smem_u32(&s_ifull[slot]));
      __syncwarp();
      if (lane == 0) arrive_warp(smem_u32(&s_ifull[slot]));
    };
    int ord = next_query(0);
    int islot = 0;
    uint32_t iuse[2] = {0u, 0u};
    if (ord >= 0) fetch_idx(ord, 0);
    while (alive && ord >= 0) {
      const int row = T_cap - 1 - (blockIdx.x + ord * gridDim.x);  // latest rows first
      const int b = seq_of(row);
      const int t = row - s_cu[b];
      const int p0 = s_p0[b];
      const int nvis = (t + p0 + 1) / r;
      const int cmp0 = s_cc[b];
      // the next query's index row is copied while this one is produced
      const int ord_next = next_query(ord + 1);
      const int cur = islot;
      if (ord_next >= 0) fetch_idx(ord_next, cur ^ 1);
      islot ^= 1;
      ord = ord_next;
      const bool okf = mbar_wait_bounded(smem_u32(&s_ifull[cur]), iuse[cur] & 1u, status);
      ++iuse[cur];
      if (bar_or(1, kProdThreads, !okf || *abort_flag != 0)) { *abort_flag = 1; alive = false; break; }
      const int32_t* src = reinterpret_cast<const int32_t*>(smem_gen + kIdxOff + (size_t)cur * k_pad * 4);
      // the query's tiles: up to the last valid slot (both warps compute the same)
      int last = -1, cnt = 0;
      for (int sl = lane; sl < k_pad; sl += 32) {
        const int g = src[sl];
        const bool ok = g >= 0 && g >= cmp0 && g < cmp0 + nvis && g < cmp_limit;
        if (g >= 0 && !ok && resolver) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
        if (ok) { last = sl; ++cnt; }
      }
      last = __reduce_max_sync(0xffffffffu, last);
      cnt = __reduce_add_sync(0xffffffffu, cnt);
      named_sync(1, kProdThreads);  // both warps are done scanning the slot before either refills it
      if (last < 0) continue;  // empty C_t: the fill kernel wrote this row
      const int ntl = last / kTK + 1;
      const uint32_t qs = nq & 1u;
      bool ok = true;
      if (resolver) {  // the query's record for the compute warps
        ok = mbar_wait_bounded(bar_rempty + 8 * qs, ((nq >> 1) & 1u) ^ 1u, status);
        if (ok && lane == 0) {
          s_qrec[qs] = QueryRec{row, ntl, cnt};
          mbar_arrive(bar_rfull + 8 * qs);
        }
      }
      // Q (64 heads x 128 dims) and qI (8 heads x 64 dims) into query slot qs
      ok = ok && mbar_wait_bounded(bar_qempty + 8 * qs, ((nq >> 1) & 1u) ^ 1u, status);
      // abort decisions are taken jointly by both producer warps (they share named barriers)
      if (bar_or(1, kProdThreads, !ok || *abort_flag != 0)) { *abort_flag = 1; alive = false; break; }
      {
        const uint32_t qb = base + kQOff + qs * kQBytes;
        for (int i = pw * 32 + lane; i < kNH * 16; i += kProdThreads) {
          const int h = i >> 4, c = i & 15;
          cp_async_16(qb + (c >> 3) * kQRegion + tc::sw128_offset(h, c & 7), q + ((int64_t)row * kNH + h) * kDim + c * 8);
        }
        if (pw == 0) {
          const int h = lane >> 3, c = lane & 7;   // 4 of the 8 heads per step
          for (int hh = h; hh < kHI; hh += 4)
            cp_async_16(base + kQIOff + qs * kQIBytes + tc::sw128_offset(hh, c),
                        qI + ((int64_t)row * kHI + hh) * kDI + c * 8);
        } else if (lane < 17) {  // the reference (64 floats) and w (8 bf16) for the compute warps
          const uint32_t ab = base + kAuxOff + qs * kAuxBytes;
          if (lane < 16) cp_async_16(ab + 16 * lane, lse_ref + (int64_t)row * kNH + 4 * lane);
          else cp_async_16(ab + 256, w + (int64_t)row * kHI);
        }
        arrive_cp_async(bar_qfull + 8 * qs);
        __syncwarp();
        if (lane == 0) arrive_warp(bar_qfull + 8 * qs);
      }
      ++nq;
      for (int pass = 0; pass < (kKeep ? 1 : 2) && alive; ++pass) {
        for (int it = 0; it < ntl; ++it, ++n) {
          const uint32_t st = n % kStages;
          bool okw = mbar_wait_bounded(bar_empty + 8 * st, ((n / kStages) & 1u) ^ 1u, status);
          if (resolver && __all_sync(0xffffffffu, okw)) {  // uniform over the warp (the ballots below)
            uint32_t m4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int sl = it * kTK + 32 * i + lane;
              int rr = -1;
              if (sl < k_pad) {
                const int g = src[sl];
                if (g >= cmp0 && g < cmp0 + nvis && g < cmp_limit) rr = g;
              }
              s_rows[st][32 * i + lane] = rr;
              m4[i] = __ballot_sync(0xffffffffu, rr >= 0);
            }
            if (lane == 0) {
              const bool p2 = kKeep || pass == 1;  // the tile carries kI (every tile with kKeep)
              const int flags = (it == 0 && pass == 0 ? kFirst : 0) | (p2 ? kPass2 : 0) |
                                (it == ntl - 1 && pass == 0 ? kLastP1 : 0) | (it == ntl - 1 && p2 ? kLast : 0);
              s_meta[st] = TileMeta{flags, {m4[0], m4[1], m4[2], m4[3]}};
            }
          }
          // one barrier: the joint abort decision, and the resolved rows are visible to every producer warp
          if (bar_or(1, kProdThreads, !okw || *abort_flag != 0)) { *abort_flag = 1; alive = false; break; }
          // coalesced gather, eight lanes per row and four rows per step: this warp takes the
          // steps j with j % kProdWarps == pw
          const uint32_t kb = base + kStageOff + st * kStageBytes;
          const int c = lane & 7, sub = lane >> 3;
#pragma unroll 2
          for (int j = pw; j < kTK / 4; j += kProdWarps) {
            const int key = 4 * j + sub;
            const int rk = s_rows[st][key];
            const __nv_bfloat16* ks = k_cmp + (int64_t)(rk < 0 ? 0 : rk) * kDim + c * 8;
            const uint32_t dst = kb + tc::sw128_offset(key, c);
            cp_async_16_zfill(dst, ks, rk >= 0);
            cp_async_16_zfill(dst + kKRegion, ks + 64, rk >= 0);
            if (kKeep || pass == 1)
              cp_async_16_zfill(dst + 2 * kKRegion, kI + (int64_t)(rk < 0 ? 0 : rk) * kDI + c * 8, rk >= 0);
          }
          arrive_cp_async(bar_full + 8 * st);
          __syncwarp();
          if (lane == 0) arrive_warp(bar_full + 8 * st);  // release: publishes s_meta
        }
      }
    }
    if (alive && pw == 0) {  // end-of-stream marker
      const uint32_t st = n % kStages;
      bool okw = mbar_wait_bounded(bar_empty + 8 * st, ((n / kStages) & 1u) ^ 1u, status);
      const uint32_t qs = nq & 1u;
      okw = okw && mbar_wait_bounded(bar_rempty + 8 * qs, ((nq >> 1) & 1u) ^ 1u, status);
      if (__any_sync(0xffffffffu, !okw)) {
        *abort_flag = 1;
      } else if (lane == 0) {
        s_meta[st] = TileMeta{kDone, {0u, 0u, 0u, 0u}};
        s_qrec[qs] = QueryRec{-1, 0, 0};
        mbar_arrive(bar_rfull + 8 * qs);
        // the full barrier expects both warps' arrivals: this warp gives all 128
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar_full + 8 * st), "r"(2 * kProdThreads)
                     : "memory");
      }
    }
    cp_async_wait<0>();
  } else if (warp >= kMmaWarp) {
    // ============ MMA issuer: S^T (both passes) and I^T (pass 2) per tile ============
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kSideRegs));
    if (warp == kMmaWarp && lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16(kTK, kNH, 0, 0);
      constexpr uint32_t kIdI = tc::idesc_bf16(kTK, 16, 0, 0);
      uint32_t n = 0, nq = 0;
      uint32_t slot = 0;               // kKeep: the tile's slot in its query's score set
      uint32_t uses[kBufs] = {0u, 0u, 0u, 0u};
      while (true) {
        const uint32_t st = n % kStages;
        if (!mbar_wait_bounded(bar_full + 8 * st, (n / kStages) & 1u, status)) { *abort_flag = 1; break; }
        const TileMeta mt = s_meta[st];
        if (mt.flags & kDone) break;
        if (*abort_flag) break;
        const uint32_t qs = nq & 1u;
        if ((mt.flags & kFirst) && !mbar_wait_bounded(bar_qfull + 8 * qs, (nq >> 1) & 1u, status)) {
          *abort_flag = 1;
          break;
        }
        uint32_t d;
        if constexpr (kKeep) {
          if (mt.flags & kFirst) {
            slot = 0;
            // the previous query's score set was read by both compute warpgroups
            if (nq > 0 && !mbar_wait_bounded(smem_u32(&s_setfree), (nq - 1) & 1u, status)) {
              *abort_flag = 1;
              break;
            }
          }
          d = slot++;
          ++uses[d];
        } else {
          d = n % kBufs;
          // the score buffer was read by the warpgroup that took tile n - kBufs
          if (n >= kBufs && !mbar_wait_bounded(bar_sfree + 8 * d, ((n / kBufs) - 1) & 1u, status)) {
            *abort_flag = 1;
            break;
          }
        }
        s_bmeta[d] = mt;                 // for the warpgroup that reads buffer d,
        mbar_arrive(bar_sfull + 8 * d);  // released by this arrival (the commit gives the other)
        tc::fence_after_sync();
        const uint32_t st_addr = base + kStageOff + st * kStageBytes;
        const uint32_t qa = base + kQOff + qs * kQBytes;
#pragma unroll
        for (int ks = 0; ks < kDim / 16; ++ks) {
          const uint64_t a = tc::smem_desc_sw128(st_addr + (ks >> 2) * kKRegion + (ks & 3) * 32, 16, 1024);
          const uint64_t bq = tc::smem_desc_sw128(qa + (ks >> 2) * kQRegion + (ks & 3) * 32, 16, 1024);
          tc::mma_bf16(tmem + d * kBufCols, a, bq, kIdS, ks > 0 ? 1u : 0u);
        }
        if (mt.flags & kPass2) {
          const uint32_t qia = base + kQIOff + qs * kQIBytes;
#pragma unroll
          for (int ks = 0; ks < kDI / 16; ++ks) {
            const uint64_t a = tc::smem_desc_sw128(st_addr + 2 * kKRegion + ks * 32, 16, 1024);
            const uint64_t bq = tc::smem_desc_sw128(qia + ks * 32, 16, 1024);
            tc::mma_bf16(tmem + kIdxCol + d * 16, a, bq, kIdI, ks > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit(bar_sfull + 8 * d);
        tc::mma_commit(bar_empty + 8 * st);
        if (mt.flags & kLast) {
          tc::mma_commit(bar_qempty + 8 * qs);  // Q / qI of this query are no longer read
          ++nq;
        }
        ++n;
      }
      // every MMA this thread issued has completed before tensor memory is freed (also after an abort)
      tc::mma_commit(smem_u32(&s_drain));
      mbar_wait_bounded(smem_u32(&s_drain), 0, status);
    }
  } else {
    // ============ compute warpgroups: warpgroup wg takes the tiles n with n % 2 == wg ============
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kComputeRegs));
    const int wg = warp >> 2, quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
    uint32_t n = 0, nq = 0;
    uint32_t uses[kBufs] = {0u, 0u, 0u, 0u};  // kKeep: queries that used each slot before this one
    while (true) {
      const uint32_t qs = nq & 1u;
      const bool okr = mbar_wait_bounded(bar_rfull + 8 * qs, (nq >> 1) & 1u, status);
      if (bar_or(2, kComputeThreads, !okr || *abort_flag != 0)) { *abort_flag = 1; break; }
      const QueryRec rec = s_qrec[qs];
      if (rec.row < 0) break;
      const int row = rec.row, ntl = rec.ntl;
      // the reference and w arrive with the query's Q (copied by the producer)
      const bool okq = mbar_wait_bounded(bar_qfull + 8 * qs, (nq >> 1) & 1u, status);
      if (bar_or(2, kComputeThreads, !okq || *abort_flag != 0)) { *abort_flag = 1; break; }
      {
        const uint8_t* ab = smem_raw + (base - smem_u32(smem_raw)) + kAuxOff + qs * kAuxBytes;
        if (tid < kNH) s_ref[tid] = -reinterpret_cast<const float*>(ab)[tid] * kLog2e;
        if (tid < kHI) s_w[tid] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(ab + 256)[tid]);
      }
      named_sync(2, kComputeThreads);
      if (tid == 0) mbar_arrive(bar_qempty + 8 * qs);  // this slot's reference and w are read
      bool failed = false;
      // ---- pass 1: Z_h = sum_j exp2(s_hj * c - r_h) ----
      float zp[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) zp[h] = 0.f;
      float tmax = -INFINITY;
      for (int it = 0; it < ntl; ++it) {
        const uint32_t nn = n + it, d = kKeep ? (uint32_t)it : nn % kBufs;
        if ((int)(d & 1u) != wg || failed) continue;
        const uint32_t par = kKeep ? (uses[d] & 1u) : ((nn / kBufs) & 1u);
        if (!mbar_wait_bounded(bar_sfull + 8 * d, par, status)) { failed = true; continue; }
        tc::fence_after_sync();
        float x[kNH];
        {
          uint32_t rs[64];
          tc::tmem_ld64_sync(tmem + lane_off + d * kBufCols, rs);
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(rs[j]);
        }
        const bool valid = (s_bmeta[d].mask[quad] >> lane) & 1u;
        if constexpr (!kKeep) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_sfree + 8 * d);
        }
        if (valid) {
#pragma unroll
          for (int h4 = 0; h4 < kNH / 4; ++h4) {
            const float4 r4 = reinterpret_cast<const float4*>(s_ref)[h4];
            float a0, a1, a2, a3;
            f2_unpack(f2_fma(f2_pack(x[4 * h4], x[4 * h4 + 1]), sc2, f2_pack(r4.x, r4.y)), a0, a1);
            f2_unpack(f2_fma(f2_pack(x[4 * h4 + 2], x[4 * h4 + 3]), sc2, f2_pack(r4.z, r4.w)), a2, a3);
            tmax = fmaxf(tmax, fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)));
            zp[4 * h4] += ex2(fminf(a0, 64.f));
            zp[4 * h4 + 1] += ex2(fminf(a1, 64.f));
            zp[4 * h4 + 2] += ex2(fminf(a2, 64.f));
            zp[4 * h4 + 3] += ex2(fminf(a3, 64.f));
          }
        }
      }
      if constexpr (!kKeep) n += ntl;
      if (tmax > 32.f) s_bad = 1;  // the reference lies far below the scores
      {
        float s0, s1;
        warp_sum64_t(zp, lane, s0, s1);
        s_z[warp][lane] = s0;
        s_z[warp][32 + lane] = s1;
      }
      if (bar_or(2, kComputeThreads, failed || *abort_flag != 0)) { *abort_flag = 1; break; }
      if (tid < kNH) {
        float z = 0.f;
#pragma unroll
        for (int ww = 0; ww < kComputeWarps; ++ww) z += s_z[ww][tid];
        const float l2 = -s_ref[tid] + __log2f(z);  // L_h in log2 units
        if (!(z > 0.f) || s_bad) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
        s_nL[tid] = z > 0.f ? -l2 : -INFINITY;
        if (teacher_lse != nullptr) teacher_lse[(int64_t)row * kNH + tid] = z > 0.f ? l2 * kLn2 : -INFINITY;
      }
      named_sync(2, kComputeThreads);
      // ---- pass 2: p(j), i_j and the KL sums ----
      float A = 0.f, Bs = 0.f, mI = -INFINITY, lI = 0.f;
      for (int it = 0; it < ntl; ++it) {
        const uint32_t nn = n + it, d = kKeep ? (uint32_t)it : nn % kBufs;
        if ((int)(d & 1u) != wg || failed) continue;
        if constexpr (!kKeep) {  // kKeep: the tile's scores are still in its slot from pass 1
          if (!mbar_wait_bounded(bar_sfull + 8 * d, (nn / kBufs) & 1u, status)) { failed = true; continue; }
          tc::fence_after_sync();
        }
        float x[kNH];
        uint32_t ri[8];
        {
          uint32_t rs[64];
          tc::tmem_ld64_ld8_sync(tmem + lane_off + d * kBufCols, tmem + lane_off + kIdxCol + d * 16, rs, ri);
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(rs[j]);
        }
        const bool valid = (s_bmeta[d].mask[quad] >> lane) & 1u;
        if constexpr (!kKeep) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_sfree + 8 * d);
        }
        if (valid) {
          uint64_t pa = f2_pack(0.f, 0.f), pb = pa;
#pragma unroll
          for (int h4 = 0; h4 < kNH / 4; ++h4) {
            const float4 L = reinterpret_cast<const float4*>(s_nL)[h4];
            float a0, a1, a2, a3;
            f2_unpack(f2_fma(f2_pack(x[4 * h4], x[4 * h4 + 1]), sc2, f2_pack(L.x, L.y)), a0, a1);
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
          for (int hh = 0; hh < kHI; ++hh) iv = fmaf(s_w[hh], fmaxf(__uint_as_float(ri[hh]), 0.f), iv);
          if (p > 0.f) A = fmaf(p, __logf(p), A);
          Bs = fmaf(p, iv, Bs);
          if (iv > mI) {
            lI = lI * __expf(mI - iv) + 1.f;
            mI = iv;
          } else {
            lI += __expf(iv - mI);
          }
        }
      }
      if constexpr (kKeep) {  // the query's score set is read: the next query's scores may overwrite it
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_setfree));
        for (int it = 0; it < ntl; ++it) ++uses[it];
      } else {
        n += ntl;
      }
      {  // reduce the per-key partials over the warp, then the eight warps
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
      if (bar_or(2, kComputeThreads, failed || *abort_flag != 0)) { *abort_flag = 1; break; }
      if (tid == 0) {
        float a = 0.f, bs = 0.f, mm = -INFINITY;
        for (int ww = 0; ww < kComputeWarps; ++ww) {
          a += s_red[ww][0];
          bs += s_red[ww][1];
          mm = fmaxf(mm, s_red[ww][2]);
        }
        float ll = 0.f;
        for (int ww = 0; ww < kComputeWarps; ++ww)
          if (s_red[ww][2] != -INFINITY) ll += s_red[ww][3] * __expf(s_red[ww][2] - mm);
        const float lse_i = mm + __logf(ll);
        kl_rows[row] = a - bs + lse_i;
        csize[row] = rec.nvalid;
        if (student_lse != nullptr) student_lse[row] = lse_i;
      }
      named_sync(2, kComputeThreads);  // s_red, s_ref and s_nL are rewritten by the next query
      if (lane == 0) mbar_arrive(bar_rempty + 8 * qs);
      ++nq;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, 512);
}

bool indexer_kl_sparse_tc_supported(const KLArgs& a, bool fp32) {
  return !fp32 && a.idx != nullptr && a.lse_cmp != nullptr && a.H == kNH && a.d == kDim && a.H_I == kHI &&
         a.d_I == kDI && a.r > 0 && a.k_pad % 4 == 0 && a.k_pad <= 4096 && a.B <= kMaxB;
}

template <bool kKeep>
static cudaError_t launch_kls(const KLArgs& a, cudaStream_t stream) {
  const size_t smem = kSmem + (size_t)8 * a.k_pad + 1024;
  auto kern = indexer_kl_sparse_tc_kernel<kKeep>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.T_cap < sms ? a.T_cap : sms;
  constexpr float kLog2e = 1.4426950408889634f;
  kern<<<grid, kThreads, smem, stream>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_cmp),
      static_cast<const __nv_bfloat16*>(a.qI), static_cast<const __nv_bfloat16*>(a.w),
      static_cast<const __nv_bfloat16*>(a.kI), a.idx, a.k_pad, a.lse_cmp, a.cu, a.cu_cmp, a.B, a.T_cap, a.r,
      a.scale * kLog2e, a.kl_rows, a.csize, a.status, a.teacher_lse, a.student_lse, a.pos0);
  return cudaGetLastError();
}

cudaError_t launch_indexer_kl_sparse_tc(const KLArgs& a, cudaStream_t stream) {
  if (a.T_cap <= 0) return cudaSuccess;
  // every row first as an empty C_t; the kernel overwrites the rows it computes
  cudaError_t err = launch_kl_zero_rows(a.kl_rows, a.csize, a.T_cap, a.teacher_lse, a.H, a.student_lse, stream);
  if (err != cudaSuccess) return err;
  // a selected set of at most kBufs tiles keeps its scores in tensor memory between the passes
  if (a.k_pad <= kBufs * kTK) return launch_kls<true>(a, stream);
  return launch_kls<false>(a, stream);
}

}  // namespace csa
