// indexer_kl_bwd_sparse_tc.cu -- backward of the selected-set (sparse-mode)
// indexer KL loss on tcgen05 tensor cores (64 heads x 128 dims, indexer 8 x 64,
// bf16), one pass over each query's selected entries with the forward's
// normalisers.
//
// "DeepSeek-V4 Attention Training Systems": §3 (L_I = sum_t KL(p_t || q_t) with
// p_t the head-averaged main-attention distribution over C_t and q_t =
// Softmax(i_{t,C_t})), §2 phase table (sparse mode: C_t is the selected set),
// §8.2 (the indexer learns through this loss only; the teacher operands are
// detached and its scores recomputed), §9 (FP32 loss math).
//
// With the per-head teacher log normaliser L_h and the student's lse_I over C_t
// kept by the KL forward, each selected entry j of query t is looked at once:
//   p(j) = (1/H) sum_h exp(scale q_h . K_j - L_h),   q(j) = exp(i_j - lse_I),
//   g_j = grad_scale (q(j) - p(j)),   C[h, j] = g_j w_h [a_hj > 0],  a_hj = qI_h . kI_j,
//   dw_h = sum_j g_j ReLU(a_hj),  dqI_h = sum_j C[h, j] kI_j,  dkI_j += sum_h C[h, j] qI_h.
// C_t is the query's own selected set, so (as in the selected-set KL forward)
// its compressed rows are gathered into 128-entry tiles; per tile
//   S^T   = K Q^T       M=128 entries, N=64 heads, K=128 dims
//   I^T   = kI qI^T     M=128 entries, N=16 (8 indexer heads + 8 zero rows), K=64 dims
//   dqI^T += kI^T C^T   M=128 (dims; the upper 64 rows unused), N=64 (8 used), K=128 entries
//   dkI   = C^T qI      M=128 entries, N=64 dims, K=16 (8 heads + 8 zero columns)
// C^T is a bf16 tile [entry][head] (columns 8..63 zero) that the compute
// threads write: the K-major A operand of dkI and the MN-major B operand of
// dqI^T.  dqI^T accumulates in tensor memory over the query's tiles; each dkI
// tile is added to the float32 gradient rows of the gathered entries with
// red.global.add by the warpgroup that computed it, read in the 16x256b shape
// so that every reduction instruction fills whole 32-byte sectors.  Three
// gathered tiles are in flight when the index rows leave room, else two.  The
// MMA warp issues a tile's gradient products after the next tile's scores, so
// the compute warpgroups never wait on their own products -- except for a
// query's last tile, whose products (and the query's dqI^T) go out at once.
// Warp roles: six producer warps (warp 8 resolves the index slots; all six
// gather rows with coalesced 16-byte cp.async copies), one MMA warp (warp 14),
// two compute warpgroups (warps 0-7) that take alternate tiles.  Every wait
// is bounded (CSA_ERR_DEVICE_TIMEOUT and a uniform abort).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "ws_sync.cuh"

namespace csa {

namespace {

using namespace ws;

constexpr int kNH = 64, kDim = 128, kHI = 8, kDI = 64;
constexpr int kTK = 128;                               // entries per tile
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
constexpr uint32_t kAuxBytes = 512;                    // per query slot: teacher normalisers (64 floats) + w (8 bf16)
constexpr uint32_t kKRegion = kTK * 128;               // 16 KB: 128 entries x 64 dims
constexpr uint32_t kCBytes = kTK * 128;                // C^T tile: 128 entries x 64 bf16 columns
// A stage is [kI | K (two 64-dim regions)]: the dqI^T product reads kI^T as a
// 128-row MN-major operand whose unused upper 64 rows then fall on the K
// regions of the same stage (inside the allocation; those rows are never read).
constexpr uint32_t kStageBytes = 3 * kKRegion;
constexpr uint32_t kQOff = 0;                          // [2 slots]
constexpr uint32_t kQIOff = 2 * kQBytes;               // [2 slots]
constexpr uint32_t kAuxOff = kQIOff + 2 * kQIBytes;    // [2 slots]
constexpr uint32_t kCOff = kAuxOff + 1024;             // [2 buffers], 1024-aligned
constexpr uint32_t kStageOff = kCOff + 2 * kCBytes;    // [stages], then [2 slots][k_pad] index rows
static_assert(kCOff % 1024 == 0 && kStageOff % 1024 == 0, "swizzle atom alignment");

// tensor memory: per buffer b (= tile parity, = the warpgroup that reads it)
constexpr uint32_t kColS = 0;      // S^T: columns 64 b .. 64 b + 63
constexpr uint32_t kColI = 128;    // I^T: columns 128 + 16 b .. (8 used)
constexpr uint32_t kColKI = 256;   // dkI: columns 256 + 64 b .. 256 + 64 b + 63
constexpr uint32_t kColDQ = 384;   // dqI^T: 64 columns (lanes 0-63 are the dims, columns 0-7 the heads)
constexpr int kMaxB = 256;         // sequences whose offsets are kept on chip

enum : int { kFirst = 1, kLast = 2, kDone = 4 };

struct TileMeta {
  int flags;
  uint32_t mask[4];  // valid entries of the tile (bit = entry % 32 of word entry / 32)
};

struct QueryRec {
  int row;       // packed row of the query
  int ntl;       // tiles
};

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void red_add_v2(float* p, uint32_t a, uint32_t b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};\n" ::"l"(p), "f"(__uint_as_float(a)), "f"(__uint_as_float(b))
               : "memory");
}

}  // namespace

// kStages: gathered tiles in flight (3 when the index rows leave room, else 2).
template <int kStages>
__global__ void __launch_bounds__(kThreads, 1)
indexer_kl_bwd_sparse_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cmp,
                                const __nv_bfloat16* __restrict__ qI, const __nv_bfloat16* __restrict__ w,
                                const __nv_bfloat16* __restrict__ kI, const int32_t* __restrict__ idx, int k_pad,
                                const float* __restrict__ teacher_lse, const float* __restrict__ student_lse,
                                const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_cmp, int B, int T_cap,
                                int r, float scale_log2, float grad_scale, __nv_bfloat16* __restrict__ dqI,
                                __nv_bfloat16* __restrict__ dw, float* __restrict__ dkI, int* status,
                                const int32_t* __restrict__ pos0) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
  __shared__ __align__(8) uint64_t s_sfull[2], s_sfree[2], s_cfull[2], s_cfree[2], s_kvfull[2], s_kvfree[2];
  __shared__ __align__(8) uint64_t s_qfull[2], s_qempty[2], s_rfull[2], s_rempty[2], s_dqdone, s_dqfree;
  __shared__ __align__(8) uint64_t s_ifull[2];  // a query's index row landed in its slot
  __shared__ __align__(8) uint64_t s_drain;
  __shared__ TileMeta s_meta[kStages];     // written by the resolver, per stage
  __shared__ TileMeta s_bmeta[2];          // copied by the MMA thread, per score buffer
  __shared__ int s_cu[kMaxB + 1], s_cc[kMaxB + 1], s_p0[kMaxB];  // the packing, on chip
  __shared__ QueryRec s_qrec[2];
  __shared__ int s_rows[kStages][kTK];
  __shared__ __align__(16) float s_nL[kNH];   // -L_h, log2 units
  __shared__ float s_w[kHI];
  __shared__ float s_lseI;
  __shared__ float s_dw[kComputeWarps][kHI];
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr uint32_t kIdxOff = kStageOff + kStages * kStageBytes;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t bar_full = smem_u32(&s_full[0]), bar_empty = smem_u32(&s_empty[0]);
  const uint32_t bar_sfull = smem_u32(&s_sfull[0]), bar_sfree = smem_u32(&s_sfree[0]);
  const uint32_t bar_cfull = smem_u32(&s_cfull[0]), bar_cfree = smem_u32(&s_cfree[0]);
  const uint32_t bar_kvfull = smem_u32(&s_kvfull[0]), bar_kvfree = smem_u32(&s_kvfree[0]);
  const uint32_t bar_qfull = smem_u32(&s_qfull[0]), bar_qempty = smem_u32(&s_qempty[0]);
  const uint32_t bar_rfull = smem_u32(&s_rfull[0]), bar_rempty = smem_u32(&s_rempty[0]);
  const uint32_t bar_dqdone = smem_u32(&s_dqdone), bar_dqfree = smem_u32(&s_dqfree);

  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_u32(&s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 2 * kProdThreads);  // per producer warp: 32 cp.async arrivals + a release of 32
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_sfull + 8 * i, 2);       // the MMA commit + the MMA thread's release of s_bmeta
      mbar_init(bar_sfree + 8 * i, 4);       // the four warps of the warpgroup that reads the buffer
      mbar_init(bar_cfull + 8 * i, 4);       // the four warps that wrote the C^T tile
      mbar_init(bar_cfree + 8 * i, 1);
      mbar_init(bar_kvfull + 8 * i, 1);
      mbar_init(bar_kvfree + 8 * i, 4);
      mbar_init(bar_qfull + 8 * i, 2 * kProdThreads);  // Q, qI, normalisers and w copies of the producer warps
      mbar_init(bar_qempty + 8 * i, 2);      // the MMA commit after the query + the compute warps' read
      mbar_init(bar_rfull + 8 * i, 1);
      mbar_init(bar_rempty + 8 * i, kComputeWarps);
      mbar_init(smem_u32(&s_ifull[i]), 2 * kProdThreads);  // the producer warps' copies
    }
    mbar_init(bar_dqdone, 1);
    mbar_init(bar_dqfree, 2);                // the two warps that read dqI^T
    mbar_init(smem_u32(&s_drain), 1);
    fence_mbar_init();
    s_abort = 0;
  }
  // zero rows 8..15 of both qI slots (the N = 16 of I^T and the K = 16 of dkI pad
  // the 8 indexer heads) and both C^T tiles (only columns 0..7 are ever written)
  for (int i = tid; i < 2 * 8 * 8; i += kThreads) {
    const int slot = i >> 6, row = 8 + ((i >> 3) & 7), c = i & 7;
    *reinterpret_cast<uint4*>(smem_gen + kQIOff + slot * kQIBytes + tc::sw128_offset(row, c)) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  for (int i = tid; i < 2 * (int)kCBytes / 16; i += kThreads)
    *reinterpret_cast<uint4*>(smem_gen + kCOff + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
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
    // ============ producers: warp 8 resolves the slots, all six gather rows ============
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
    // copy a query's index row into slot `slot` (every producer warp, 16-byte chunks)
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
      // the query's tiles: up to the last valid slot (every warp computes the same)
      int last = -1;
      for (int sl = lane; sl < k_pad; sl += 32) {
        const int g = src[sl];
        const bool ok = g >= 0 && g >= cmp0 && g < cmp0 + nvis && g < cmp_limit;
        if (g >= 0 && !ok && resolver) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
        if (ok) last = sl;
      }
      last = __reduce_max_sync(0xffffffffu, last);
      named_sync(1, kProdThreads);  // every warp is done scanning the slot before it is refilled
      if (last < 0) continue;  // empty C_t: its gradients stay zero
      const int ntl = last / kTK + 1;
      const uint32_t qs = nq & 1u;
      bool ok = true;
      if (resolver) {  // the query's record for the compute warps
        ok = mbar_wait_bounded(bar_rempty + 8 * qs, ((nq >> 1) & 1u) ^ 1u, status);
        if (ok && lane == 0) {
          s_qrec[qs] = QueryRec{row, ntl};
          mbar_arrive(bar_rfull + 8 * qs);
        }
      }
      // Q (64 heads x 128 dims), qI (8 heads x 64 dims), the teacher's normalisers and w into slot qs
      ok = ok && mbar_wait_bounded(bar_qempty + 8 * qs, ((nq >> 1) & 1u) ^ 1u, status);
      // abort decisions are taken jointly by the producer warps (they share named barriers)
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
        } else if (pw == 1 && lane < 17) {  // the teacher's normalisers (64 floats) and w (8 bf16)
          const uint32_t ab = base + kAuxOff + qs * kAuxBytes;
          if (lane < 16) cp_async_16(ab + 16 * lane, teacher_lse + (int64_t)row * kNH + 4 * lane);
          else cp_async_16(ab + 256, w + (int64_t)row * kHI);
        }
        arrive_cp_async(bar_qfull + 8 * qs);
        __syncwarp();
        if (lane == 0) arrive_warp(bar_qfull + 8 * qs);
      }
      ++nq;
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
            const int flags = (it == 0 ? kFirst : 0) | (it == ntl - 1 ? kLast : 0);
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
          const int64_t rs = rk < 0 ? 0 : rk;
          const uint32_t dst = kb + tc::sw128_offset(key, c);
          cp_async_16_zfill(dst, kI + rs * kDI + c * 8, rk >= 0);
          cp_async_16_zfill(dst + kKRegion, k_cmp + rs * kDim + c * 8, rk >= 0);
          cp_async_16_zfill(dst + 2 * kKRegion, k_cmp + rs * kDim + 64 + c * 8, rk >= 0);
        }
        arrive_cp_async(bar_full + 8 * st);
        __syncwarp();
        if (lane == 0) arrive_warp(bar_full + 8 * st);  // release: publishes s_meta / s_rows
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
        s_qrec[qs] = QueryRec{-1, 0};
        mbar_arrive(bar_rfull + 8 * qs);
        // the full barrier expects every producer warp's arrivals: this warp gives all of them
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar_full + 8 * st), "r"(2 * kProdThreads)
                     : "memory");
      }
    }
    cp_async_wait<0>();
  } else if (warp >= kMmaWarp) {
    // ============ MMA issuer: scores of tile n, then the gradient products of tile n - 1 ============
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kSideRegs));
    if (warp == kMmaWarp && lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16(kTK, kNH, 0, 0);   // S^T = K Q^T
      constexpr uint32_t kIdI = tc::idesc_bf16(kTK, 16, 0, 0);    // I^T = kI qI^T
      constexpr uint32_t kIdDQ = tc::idesc_bf16(128, 64, 1, 1);   // dqI^T += kI^T C^T
      constexpr uint32_t kIdKI = tc::idesc_bf16(kTK, kDI, 0, 1);  // dkI = C^T qI
      uint32_t n = 0, nq = 0, nqg = 0;  // tiles, queries started, queries whose gradients are issued
      bool ok = true;
      // the tile whose gradient products are still to be issued
      bool pend = false;
      uint32_t pst = 0, pn = 0, pqs = 0;
      int pflags = 0;
      auto grad = [&]() -> bool {
        const uint32_t pb = pn & 1u;
        if (!mbar_wait_bounded(bar_cfull + 8 * pb, (pn >> 1) & 1u, status)) return false;
        if (pn >= 2 && !mbar_wait_bounded(bar_kvfree + 8 * pb, ((pn >> 1) - 1) & 1u, status)) return false;
        const bool first = (pflags & kFirst) != 0;
        if (first && nqg > 0 && !mbar_wait_bounded(bar_dqfree, (nqg - 1) & 1u, status)) return false;
        tc::fence_after_sync();
        const uint32_t sti = base + kStageOff + pst * kStageBytes;  // the tile's kI
        const uint32_t cb = base + kCOff + pb * kCBytes;
#pragma unroll
        for (int ks = 0; ks < kTK / 16; ++ks) {  // over the tile's entries, 16 at a time
          const uint64_t a = tc::smem_desc_sw128(sti + ks * 2048, kKRegion, 1024);
          const uint64_t bd = tc::smem_desc_sw128(cb + ks * 2048, 1024, 1024);
          tc::mma_bf16(tmem + kColDQ, a, bd, kIdDQ, (first && ks == 0) ? 0u : 1u);
        }
        {  // over the 16 (head) columns of C^T: the 8 heads and 8 zero columns
          const uint64_t a = tc::smem_desc_sw128(cb, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(base + kQIOff + pqs * kQIBytes, 1024, 1024);
          tc::mma_bf16(tmem + kColKI + pb * kDI, a, bd, kIdKI, 0u);
        }
        tc::mma_commit(bar_cfree + 8 * pb);
        tc::mma_commit(bar_kvfull + 8 * pb);
        tc::mma_commit(bar_empty + 8 * pst);
        if (pflags & kLast) {
          tc::mma_commit(bar_dqdone);
          tc::mma_commit(bar_qempty + 8 * pqs);  // Q / qI of this query are no longer read
          ++nqg;
        }
        return true;
      };
      while (true) {
        const uint32_t st = n % kStages, b = n & 1u;
        // a query's last tile: its products (and the query's dqI^T) go out before the next
        // tile is waited for, so the compute warps can close the query while it is gathered
        if (pend && (pflags & kLast)) {
          if (!grad()) { ok = false; break; }
          pend = false;
        }
        if (!mbar_wait_bounded(bar_full + 8 * st, (n / kStages) & 1u, status)) { ok = false; break; }
        const TileMeta mt = s_meta[st];
        if (mt.flags & kDone) break;
        if (*abort_flag) break;
        const uint32_t qs = nq & 1u;
        if ((mt.flags & kFirst) && !mbar_wait_bounded(bar_qfull + 8 * qs, (nq >> 1) & 1u, status)) {
          ok = false;
          break;
        }
        // score buffer b was read by the warpgroup that took tile n - 2
        if (n >= 2 && !mbar_wait_bounded(bar_sfree + 8 * b, ((n >> 1) - 1) & 1u, status)) { ok = false; break; }
        s_bmeta[b] = mt;                 // for the warpgroup that reads buffer b,
        mbar_arrive(bar_sfull + 8 * b);  // released by this arrival (the commit gives the other)
        tc::fence_after_sync();
        const uint32_t sa = base + kStageOff + st * kStageBytes;
        const uint32_t qa = base + kQOff + qs * kQBytes, qia = base + kQIOff + qs * kQIBytes;
#pragma unroll
        for (int ks = 0; ks < kDim / 16; ++ks) {
          const uint64_t a = tc::smem_desc_sw128(sa + kKRegion + (ks >> 2) * kKRegion + (ks & 3) * 32, 16, 1024);
          const uint64_t bq = tc::smem_desc_sw128(qa + (ks >> 2) * kQRegion + (ks & 3) * 32, 16, 1024);
          tc::mma_bf16(tmem + kColS + b * kNH, a, bq, kIdS, ks > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < kDI / 16; ++ks) {
          const uint64_t a = tc::smem_desc_sw128(sa + ks * 32, 16, 1024);
          const uint64_t bq = tc::smem_desc_sw128(qia + ks * 32, 16, 1024);
          tc::mma_bf16(tmem + kColI + b * 16, a, bq, kIdI, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar_sfull + 8 * b);
        if (pend && !grad()) { ok = false; break; }
        pend = true;
        pst = st;
        pn = n;
        pqs = qs;
        pflags = mt.flags;
        if (mt.flags & kLast) ++nq;
        ++n;
      }
      if (ok && pend && !*abort_flag) ok = grad();  // the last tile's products
      if (!ok) *abort_flag = 1;
      // every MMA this thread issued has completed before tensor memory is freed (also after an abort)
      tc::mma_commit(smem_u32(&s_drain));
      mbar_wait_bounded(smem_u32(&s_drain), 0, status);
    }
  } else {
    // ============ compute warpgroups: warpgroup wg takes the tiles n with n % 2 == wg ============
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kComputeRegs));
    const int wg = warp >> 2, quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int key = quad * 32 + lane;  // tensor-memory lane: entry of the tile
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    constexpr float kLog2e = 1.4426950408889634f;
    uint32_t n = 0, nq = 0;
    bool failed = false;
    // this warpgroup's previous tile, whose dkI rows are still to be added
    bool have_prev = false;
    uint32_t prev_n = 0;
    int prev_rk = -1;
    // dkI of tile tn for this warp's 32 entries (rk: this lane's entry's gathered
    // row, -1: none), read in the 16x256b shape so that four threads hold 32
    // contiguous bytes of a row and each reduction instruction fills whole sectors
    auto epilogue = [&](uint32_t tn, int rk) {
      const uint32_t b = tn & 1u;
      const bool okw = mbar_wait_bounded(bar_kvfull + 8 * b, (tn >> 1) & 1u, status);
      if (__any_sync(0xffffffffu, !okw)) { failed = true; return; }
      tc::fence_after_sync();
      uint32_t v[4][2][8];
#pragma unroll
      for (int cb = 0; cb < 4; ++cb)
        tc::tmem_ld16x256_pair_sync(tmem + ((uint32_t)(quad * 32) << 16) + kColKI + b * kDI + cb * 16,
                                    tmem + ((uint32_t)(quad * 32 + 16) << 16) + kColKI + b * kDI + cb * 16, v[cb][0],
                                    v[cb][1]);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_kvfree + 8 * b);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int rr = __shfl_sync(0xffffffffu, rk, hf * 16 + e * 8 + (lane >> 2));  // entry of these registers
          if (rr >= 0) {
            float* dst = dkI + (int64_t)rr * kDI + 2 * (lane & 3);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
              red_add_v2(dst + cb * 16, v[cb][hf][2 * e], v[cb][hf][2 * e + 1]);
              red_add_v2(dst + cb * 16 + 8, v[cb][hf][4 + 2 * e], v[cb][hf][4 + 2 * e + 1]);
            }
          }
        }
    };
    while (true) {
      const uint32_t qs = nq & 1u;
      const bool okr = mbar_wait_bounded(bar_rfull + 8 * qs, (nq >> 1) & 1u, status);
      if (bar_or(2, kComputeThreads, !okr || failed || *abort_flag != 0)) { *abort_flag = 1; break; }
      const QueryRec rec = s_qrec[qs];
      if (rec.row < 0) break;
      const int row = rec.row, ntl = rec.ntl;
      // the teacher's normalisers and w arrive with the query's Q (copied by the producer)
      const bool okq = mbar_wait_bounded(bar_qfull + 8 * qs, (nq >> 1) & 1u, status);
      if (bar_or(2, kComputeThreads, !okq || *abort_flag != 0)) { *abort_flag = 1; break; }
      {
        const uint8_t* ab = smem_gen + kAuxOff + qs * kAuxBytes;
        if (tid < kNH) {
          const float L = reinterpret_cast<const float*>(ab)[tid];
          s_nL[tid] = isfinite(L) ? -L * kLog2e : 0.f;
        }
        if (tid < kHI) s_w[tid] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(ab + 256)[tid]);
        if (tid == 0) s_lseI = student_lse[row];
      }
      named_sync(2, kComputeThreads);
      if (tid == 0) mbar_arrive(bar_qempty + 8 * qs);  // this slot's normalisers and w are read
      const float lseI = s_lseI;
      const bool q_ok = isfinite(lseI);
      float w_r[kHI];
#pragma unroll
      for (int h = 0; h < kHI; ++h) w_r[h] = s_w[h];
      float dwa[kHI];
#pragma unroll
      for (int h = 0; h < kHI; ++h) dwa[h] = 0.f;
      for (int it = 0; it < ntl; ++it) {
        const uint32_t nn = n + it, b = nn & 1u;
        if ((int)b != wg || failed) continue;
        if (!mbar_wait_bounded(bar_sfull + 8 * b, (nn >> 1) & 1u, status)) { failed = true; continue; }
        tc::fence_after_sync();
        float x[kNH];
        uint32_t ri[8];
        {
          uint32_t rs[64];
          tc::tmem_ld64_ld8_sync(tmem + lane_off + kColS + b * kNH, tmem + lane_off + kColI + b * 16, rs, ri);
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(rs[j]);
        }
        const bool valid = (s_bmeta[b].mask[quad] >> lane) & 1u;
        const int rk = valid ? s_rows[nn % kStages][key] : -1;  // the stage is held until this tile's products
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfree + 8 * b);
        float g = 0.f;
        if (valid && q_ok) {
          // teacher p(j): the mean over heads of exp2(s scale log2e - L_h log2e)
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
          for (int h = 0; h < kHI; ++h) iv = fmaf(w_r[h], fmaxf(__uint_as_float(ri[h]), 0.f), iv);
          g = grad_scale * (__expf(iv - lseI) - p);
        }
        // dw partials and this entry's row of C^T (bf16, heads 0..7)
        uint32_t cp[kHI / 2];
#pragma unroll
        for (int h = 0; h < kHI; h += 2) {
          const float a0 = __uint_as_float(ri[h]), a1 = __uint_as_float(ri[h + 1]);
          dwa[h] = fmaf(g, fmaxf(a0, 0.f), dwa[h]);
          dwa[h + 1] = fmaf(g, fmaxf(a1, 0.f), dwa[h + 1]);
          cp[h / 2] = pack_bf16x2(a0 > 0.f ? g * w_r[h] : 0.f, a1 > 0.f ? g * w_r[h + 1] : 0.f);
        }
        if (nn >= 2) {  // the products of this warpgroup's previous tile have read its C^T tile
          const bool okc = mbar_wait_bounded(bar_cfree + 8 * b, ((nn >> 1) - 1) & 1u, status);
          if (__any_sync(0xffffffffu, !okc)) { failed = true; continue; }
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(base + kCOff + b * kCBytes + tc::sw128_offset(key, 0)),
                     "r"(cp[0]), "r"(cp[1]), "r"(cp[2]), "r"(cp[3])
                     : "memory");
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cfull + 8 * b);
        if (have_prev) epilogue(prev_n, prev_rk);
        have_prev = true;
        prev_n = nn;
        prev_rk = rk;
      }
      n += ntl;
      // dw: the per-entry partials summed over the warp, then the eight warps
#pragma unroll
      for (int h = 0; h < kHI; ++h) {
        float v = dwa[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_dw[warp][h] = v;
      }
      if (bar_or(2, kComputeThreads, failed || *abort_flag != 0)) { *abort_flag = 1; break; }
      if (tid < kHI) {
        float v = 0.f;
        for (int ww = 0; ww < kComputeWarps; ++ww) v += s_dw[ww][tid];
        dw[(int64_t)row * kHI + tid] = __float2bfloat16_rn(v);
      }
      // dqI: dqI^T lanes 0..63 (dims) x columns 0..7 (heads), read by warps 0 and 1
      if (warp < 2) {
        const bool okd = mbar_wait_bounded(bar_dqdone, nq & 1u, status);
        if (__any_sync(0xffffffffu, !okd)) {
          failed = true;
        } else {
          tc::fence_after_sync();
          uint32_t v[8];
          tc::tmem_ld8_sync(tmem + lane_off + kColDQ, v);
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dqfree);
          const int dim = key;
#pragma unroll
          for (int h = 0; h < kHI; ++h)
            dqI[((int64_t)row * kHI + h) * kDI + dim] = __float2bfloat16_rn(__uint_as_float(v[h]));
        }
      }
      named_sync(2, kComputeThreads);  // s_dw, s_nL and s_w are rewritten by the next query
      if (lane == 0) mbar_arrive(bar_rempty + 8 * qs);
      ++nq;
    }
    if (have_prev && !failed && !*abort_flag) epilogue(prev_n, prev_rk);
    if (failed) *abort_flag = 1;
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, 512);
}

bool indexer_kl_bwd_sparse_tc_supported(const KLBwdArgs& a, bool fp32) {
  return !fp32 && a.idx != nullptr && a.lse_cmp != nullptr && a.student_lse != nullptr && a.H == kNH &&
         a.d == kDim && a.H_I == kHI && a.d_I == kDI && a.r > 0 && a.k_pad % 4 == 0 && a.k_pad <= 4096 &&
         a.B <= kMaxB;
}

template <int kStages>
static cudaError_t launch_kbs(const KLBwdArgs& a, size_t smem, cudaStream_t stream) {
  auto kern = indexer_kl_bwd_sparse_tc_kernel<kStages>;
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
      static_cast<const __nv_bfloat16*>(a.kI), a.idx, a.k_pad, a.lse_cmp, a.student_lse, a.cu, a.cu_cmp, a.B,
      a.T_cap, a.r, a.scale * kLog2e, a.grad_scale, static_cast<__nv_bfloat16*>(a.dqI),
      static_cast<__nv_bfloat16*>(a.dw), a.dkI, a.status, a.pos0);
  return cudaGetLastError();
}

cudaError_t launch_indexer_kl_bwd_sparse_tc(const KLBwdArgs& a, cudaStream_t stream) {
  if (a.T_cap <= 0) return cudaSuccess;
  // rows without a selected entry (and capacity rows) keep zero gradients
  cudaError_t err = cudaMemsetAsync(a.dkI, 0, (size_t)a.n_cmp_cap * kDI * 4, stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(a.dqI, 0, (size_t)a.T_cap * kHI * kDI * 2, stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(a.dw, 0, (size_t)a.T_cap * kHI * 2, stream);
  if (err != cudaSuccess) return err;
  // a third stage when it fits beside the index rows (227 KB a block, less 8 KB of static arrays)
  const size_t idx_bytes = (size_t)8 * a.k_pad + 1024;
  const size_t smem3 = kStageOff + 3 * (size_t)kStageBytes + idx_bytes;
  if (smem3 + 8 * 1024 <= 232448) return launch_kbs<3>(a, smem3, stream);
  return launch_kbs<2>(a, kStageOff + 2 * (size_t)kStageBytes + idx_bytes, stream);
}

}  // namespace csa
