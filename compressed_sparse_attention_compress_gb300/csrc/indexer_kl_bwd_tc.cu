// indexer_kl_bwd_tc.cu -- backward of the dense-teacher indexer KL loss on
// tcgen05 tensor cores (64 heads x 128 dims, indexer 8 x 64, bf16), one pass
// over the keys with the forward's normalisers.
//
// "DeepSeek-V4 Attention Training Systems": §3 (L_I = sum_t KL(p_t || q_t) with
// p_t the head-averaged main-attention distribution over C_t and q_t =
// Softmax(i_{t,C_t})), §8.2 (the indexer learns through this loss only; the
// teacher operands are detached and its scores recomputed), §9 (FP32 loss
// math).
//
// With the per-head teacher log-sum-exp lse_h and the student's lse_I over C_t
// kept by the KL forward, each (query, entry) pair is looked at once:
//   p(j) = (1/H) sum_h exp(scale q_h . K_j - lse_h),   q(j) = exp(i_j - lse_I),
//   g_j = grad_scale (q(j) - p(j)),   C[h, j] = g_j w_h [a_hj > 0],  a_hj = qI_h . kI_j,
//   dw_h = sum_j g_j ReLU(a_hj),  dqI_h = sum_j C[h, j] kI_j,  dkI_j = sum_h C[h, j] qI_h.
// C_t is a prefix of the sequence's compressed rows, so, as in the forward, a
// CTA takes a block of 4 consecutive queries and streams the prefix through
// shared memory in tiles of 128 entries (TMA, 128-byte swizzle):
//   S^T   = K Q^T       M=128 entries, N=256 (4 queries x 64 heads), K=128 dims
//   I^T   = kI qI^T     M=128 entries, N=32 (4 queries x 8 heads),  K=64 dims
//   dqI^T += kI^T C^T   M=128 (dims; the upper 64 rows unused), N=64 (32 used), K=128 entries
//   dkI   = C^T qI      M=128 entries, N=64 dims, K=32
// C^T is one bf16 tile [entry][(query, head)] (columns 32..63 zero) written by
// the compute threads: the K-major A operand of dkI and the MN-major B operand
// of dqI^T.  dqI^T accumulates in tensor memory over the block; each dkI tile
// (two tensor-memory buffers) is added to the float32 gradient rows with
// red.global.add by the compute threads while the next tile's scores run.
// Each block visits its tiles in an order rotated by its position, so that
// concurrent blocks add to different rows while a query's gradients stay
// independent of how the rows are packed or split.
// Warps 0-15 compute (warpgroup = query, thread = entry of the tile), warp 16
// issues the TMA loads, warp 17 allocates tensor memory and issues the MMAs.
// Every wait is bounded (CSA_ERR_DEVICE_TIMEOUT and a uniform abort).
#include <math.h>

#include "common.cuh"
#include "kl_blocks.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace csa {

namespace {

constexpr int kQB = 4;          // queries per block
constexpr int kNH = 64;         // heads
constexpr int kDim = 128;       // head dim
constexpr int kHI = 8;          // indexer heads
constexpr int kDI = 64;         // indexer head dim
constexpr int kTK = 128;        // entries per tile
constexpr int kKStages = 3;     // K tiles: free once S^T is issued
constexpr int kIStages = 2;     // kI tiles: free once dqI^T is issued
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kProdWarp = kComputeWarps, kMmaWarp = kComputeWarps + 1;
constexpr int kThreads = kComputeThreads + 64;

constexpr uint32_t kQRegion = kQB * kNH * 128;        // 32 KB: 256 rows x 64 dims
constexpr uint32_t kQOff = 0;
constexpr uint32_t kQIOff = 2 * kQRegion;             // 4 KB: 32 rows x 64 dims
constexpr uint32_t kKRegion = kTK * 128;              // 16 KB: 128 rows x 64 dims
constexpr uint32_t kKStage = 2 * kKRegion;
constexpr uint32_t kKOff = kQIOff + 4096;
constexpr uint32_t kIOff = kKOff + kKStages * kKStage;
constexpr uint32_t kCOff = kIOff + kIStages * kKRegion;  // C^T tile [entry][64] bf16
constexpr uint32_t kSmemBytes = kCOff + kTK * 128;       // 212 KB
static_assert(kKOff % 1024 == 0 && kIOff % 1024 == 0 && kCOff % 1024 == 0, "swizzle atom alignment");
// dqI^T reads kI^T as a 128-row MN-major operand: its second 64-row half lies
// one region past the kI tile (the next kI stage or the C^T tile), inside the
// allocation; those accumulator rows are never read.
static_assert(kIOff + kIStages * kKRegion + kKRegion <= kSmemBytes, "dqI^T upper half stays in shared memory");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S^T: 256 columns
constexpr uint32_t kColI = 256;   // I^T: 32 columns
constexpr uint32_t kColDQ = 320;  // dqI^T: 64 columns (lanes 0..63 used)
constexpr uint32_t kColKI = 384;  // dkI: two buffers of 64 columns

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void red_add_v2(float* p, uint32_t a, uint32_t b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};\n" ::"l"(p), "f"(__uint_as_float(a)), "f"(__uint_as_float(b))
               : "memory");
}

__device__ __forceinline__ int rotated_tile(int ii, int rot, int ntiles) {
  const int ti = ii + rot;
  return ti >= ntiles ? ti - ntiles : ti;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
indexer_kl_bwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_qi, const __grid_constant__ CUtensorMap map_ki,
                         const __nv_bfloat16* __restrict__ w, const float* __restrict__ teacher_lse,
                         const float* __restrict__ student_lse, const int32_t* __restrict__ cu,
                         const int32_t* __restrict__ cu_cmp, int B, int r, float scale_log2, float grad_scale,
                         __nv_bfloat16* __restrict__ dqI, __nv_bfloat16* __restrict__ dw, float* __restrict__ dkI,
                         int* status, const int32_t* __restrict__ pos0) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_kfull[kKStages], s_kempty[kKStages], s_ifull[kIStages], s_iempty[kIStages];
  __shared__ __align__(8) uint64_t s_sfull, s_sfree, s_cfull, s_cfree, s_kvfull[2], s_kvfree[2];
  __shared__ __align__(8) uint64_t s_qfull, s_qempty, s_dqdone, s_dqfree;
  __shared__ __align__(8) uint64_t s_drain;  // the MMA thread's last commit, before tensor memory is freed
  __shared__ __align__(16) float s_L[kQB][kNH];  // per (query, head): minus the teacher lse, log2 units
  __shared__ float s_w[kQB][kHI];
  __shared__ float s_lseI[kQB];
  __shared__ float s_dw[kComputeWarps][kHI];
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_kfull = smem_u32(&s_kfull[0]), bar_kempty = smem_u32(&s_kempty[0]);
  const uint32_t bar_ifull = smem_u32(&s_ifull[0]), bar_iempty = smem_u32(&s_iempty[0]);
  const uint32_t bar_sfull = smem_u32(&s_sfull), bar_sfree = smem_u32(&s_sfree);
  const uint32_t bar_cfull = smem_u32(&s_cfull), bar_cfree = smem_u32(&s_cfree);
  const uint32_t bar_kvfull = smem_u32(&s_kvfull[0]), bar_kvfree = smem_u32(&s_kvfree[0]);
  const uint32_t bar_qfull = smem_u32(&s_qfull), bar_qempty = smem_u32(&s_qempty);
  const uint32_t bar_dqdone = smem_u32(&s_dqdone), bar_dqfree = smem_u32(&s_dqfree);

  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
    }
    for (int s = 0; s < kIStages; ++s) {
      mbar_init(bar_ifull + 8 * s, 1);
      mbar_init(bar_iempty + 8 * s, 1);
    }
    mbar_init(bar_sfull, 1);
    mbar_init(bar_sfree, kComputeWarps);
    mbar_init(bar_cfull, kComputeWarps);
    mbar_init(bar_cfree, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_kvfull + 8 * s, 1);
      mbar_init(bar_kvfree + 8 * s, kComputeWarps);
    }
    mbar_init(bar_qfull, 1);
    mbar_init(bar_qempty, 1);
    mbar_init(bar_dqdone, 1);
    mbar_init(bar_dqfree, 2);  // the two warps that read dqI^T
    mbar_init(smem_u32(&s_drain), 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (tid < kComputeThreads) {  // the C^T tile starts zero (columns 32..63 stay zero)
    const uint32_t p = base + kCOff + tid * 32;
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};\n" ::"r"(p), "r"(0u) : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};\n" ::"r"(p + 16), "r"(0u) : "memory");
    tc::fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int total = klb::total_blocks<kQB>(cu, B);
  volatile int* abort_flag = &s_abort;

  if (warp == kProdWarp) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_qi);
      tma_prefetch_map(&map_ki);
      uint32_t t = 0, nblk = 0;
      for (int k = blockIdx.x; k < total && !*abort_flag; k += gridDim.x) {
        klb::Block bk;
        if (!klb::block_of<kQB, kTK>(cu, cu_cmp, B, r, total, k, bk, pos0) || bk.ntiles == 0) continue;
        if (!mbar_wait_bounded(bar_qempty, (nblk & 1u) ^ 1u, status)) { *abort_flag = 1; break; }
        ++nblk;
        mbar_arrive_expect_tx(bar_qfull, 2 * kQRegion + kQB * kHI * 128);
        for (int rg = 0; rg < 2; ++rg)
          for (int m = 0; m < 2; ++m)
            tma_load_2d(base + kQOff + rg * kQRegion + m * 16384, &map_q, rg * 64, (bk.seq0 + bk.q0) * kNH + m * 128,
                        bar_qfull);
        tma_load_2d(base + kQIOff, &map_qi, 0, (bk.seq0 + bk.q0) * kHI, bar_qfull);
        const int rot = ((bk.q0 + bk.p0) / kQB) % bk.ntiles;  // by position: results do not depend on the packing
        for (int ii = 0; ii < bk.ntiles; ++ii, ++t) {
          const int row = bk.cmp0 + rotated_tile(ii, rot, bk.ntiles) * kTK;
          const uint32_t sk = t % kKStages, si = t % kIStages;
          if (!mbar_wait_bounded(bar_kempty + 8 * sk, ((t / kKStages) & 1u) ^ 1u, status)) { *abort_flag = 1; break; }
          const uint32_t stk = base + kKOff + sk * kKStage;
          mbar_arrive_expect_tx(bar_kfull + 8 * sk, kKStage);
          tma_load_2d(stk, &map_k, 0, row, bar_kfull + 8 * sk);
          tma_load_2d(stk + kKRegion, &map_k, 64, row, bar_kfull + 8 * sk);
          if (!mbar_wait_bounded(bar_iempty + 8 * si, ((t / kIStages) & 1u) ^ 1u, status)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(bar_ifull + 8 * si, kKRegion);
          tma_load_2d(base + kIOff + si * kKRegion, &map_ki, 0, row, bar_ifull + 8 * si);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16(kTK, kQB * kNH, 0, 0);   // S^T = K Q^T
      constexpr uint32_t kIdI = tc::idesc_bf16(kTK, kQB * kHI, 0, 0);   // I^T = kI qI^T
      constexpr uint32_t kIdDQ = tc::idesc_bf16(128, 64, 1, 1);         // dqI^T += kI^T C^T
      constexpr uint32_t kIdKI = tc::idesc_bf16(kTK, kDI, 0, 1);        // dkI = C^T qI
      uint32_t t = 0, nblk = 0;
      bool ok = true;
      // the gradient products of tile tg (its C^T tile written by the compute threads)
      auto grad = [&](uint32_t tg, bool first) -> bool {
        const uint32_t si = tg % kIStages, buf = tg & 1u;
        if (!mbar_wait_bounded(bar_cfull, tg & 1u, status)) return false;
        if (tg >= 2 && !mbar_wait_bounded(bar_kvfree + 8 * buf, ((tg >> 1) - 1) & 1u, status)) return false;
        if (first && nblk > 0 && !mbar_wait_bounded(bar_dqfree, (nblk - 1) & 1u, status)) return false;
        tc::fence_after_sync();
        const uint32_t sti = base + kIOff + si * kKRegion;
#pragma unroll
        for (int ks = 0; ks < kTK / 16; ++ks) {  // over the tile's entries, 16 at a time
          const uint64_t a = tc::smem_desc_sw128(sti + ks * 2048, kKRegion, 1024);
          const uint64_t b = tc::smem_desc_sw128(base + kCOff + ks * 2048, 1024, 1024);
          tc::mma_bf16(tmem + kColDQ, a, b, kIdDQ, (first && ks == 0) ? 0u : 1u);
        }
#pragma unroll
        for (int ks = 0; ks < (kQB * kHI) / 16; ++ks) {  // over the block's (query, head) pairs
          const uint64_t a = tc::smem_desc_sw128(base + kCOff + ks * 32, 16, 1024);
          const uint64_t b = tc::smem_desc_sw128(base + kQIOff + ks * 2048, 1024, 1024);
          tc::mma_bf16(tmem + kColKI + buf * kDI, a, b, kIdKI, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar_cfree);
        tc::mma_commit(bar_kvfull + 8 * buf);
        tc::mma_commit(bar_iempty + 8 * si);
        return true;
      };
      for (int k = blockIdx.x; k < total && ok && !*abort_flag; k += gridDim.x) {
        klb::Block bk;
        if (!klb::block_of<kQB, kTK>(cu, cu_cmp, B, r, total, k, bk, pos0) || bk.ntiles == 0) continue;
        if (!mbar_wait_bounded(bar_qfull, nblk & 1u, status)) { ok = false; break; }
        for (int ii = 0; ii < bk.ntiles; ++ii, ++t) {
          const uint32_t sk = t % kKStages, si = t % kIStages;
          if (!mbar_wait_bounded(bar_kfull + 8 * sk, (t / kKStages) & 1u, status) ||
              !mbar_wait_bounded(bar_ifull + 8 * si, (t / kIStages) & 1u, status) ||
              (t > 0 && !mbar_wait_bounded(bar_sfree, (t - 1) & 1u, status))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t stk = base + kKOff + sk * kKStage;
#pragma unroll
          for (int ks = 0; ks < kDim / 16; ++ks) {
            const uint64_t a = tc::smem_desc_sw128(stk + (ks >> 2) * kKRegion + (ks & 3) * 32, 16, 1024);
            const uint64_t b = tc::smem_desc_sw128(base + kQOff + (ks >> 2) * kQRegion + (ks & 3) * 32, 16, 1024);
            tc::mma_bf16(tmem + kColS, a, b, kIdS, ks > 0 ? 1u : 0u);
          }
          const uint32_t sti = base + kIOff + si * kKRegion;
#pragma unroll
          for (int ks = 0; ks < kDI / 16; ++ks) {
            const uint64_t a = tc::smem_desc_sw128(sti + ks * 32, 16, 1024);
            const uint64_t b = tc::smem_desc_sw128(base + kQIOff + ks * 32, 16, 1024);
            tc::mma_bf16(tmem + kColI, a, b, kIdI, ks > 0 ? 1u : 0u);
          }
          tc::mma_commit(bar_sfull);
          tc::mma_commit(bar_kempty + 8 * sk);
          if (ii > 0 && !grad(t - 1, ii == 1)) { ok = false; break; }
        }
        if (!ok || !grad(t - 1, bk.ntiles == 1)) { ok = false; break; }
        tc::mma_commit(bar_dqdone);
        tc::mma_commit(bar_qempty);  // Q / qI free once this block's MMAs are done
        ++nblk;
      }
      if (!ok) *abort_flag = 1;
      // every MMA this thread issued has completed before tensor memory is freed (also after an abort)
      tc::mma_commit(smem_u32(&s_drain));
      mbar_wait_bounded(smem_u32(&s_drain), 0, status);
    }
  } else {
    // ---------------- compute: warpgroup q = query, thread = entry of the tile ----------------
    const int q = warp >> 2;                 // query of the block
    const int quad = warp & 3;               // tensor-memory lane quadrant
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int rowl = quad * 32 + lane;       // tensor-memory lane: entry of the tile
    constexpr float kLog2e = 1.4426950408889634f;
    uint32_t t = 0, nblk = 0;
    // the dkI epilogue of tile tp: rows row0 + [0, nvalid) of the gradient,
    // this warpgroup's 16 dims, this warp's 32 lanes as two 16-lane halves
    auto epilogue = [&](uint32_t tp, int64_t row0, int nvalid) -> bool {
      const uint32_t buf = tp & 1u;
      const bool okw = mbar_wait_bounded(bar_kvfull + 8 * buf, (tp >> 1) & 1u, status);
      if (__any_sync(0xffffffffu, !okw)) return false;
      tc::fence_after_sync();
      uint32_t v[2][8];
      tc::tmem_ld16x256_pair_sync(tmem + ((uint32_t)(quad * 32) << 16) + kColKI + buf * kDI + q * 16,
                                  tmem + ((uint32_t)(quad * 32 + 16) << 16) + kColKI + buf * kDI + q * 16, v[0], v[1]);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_kvfree + 8 * buf);
      const int c = q * 16 + 2 * (lane & 3);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int rl = quad * 32 + hf * 16 + e * 8 + (lane >> 2);  // lane of the tile = entry
          if (rl < nvalid) {
            float* dst = dkI + (row0 + rl) * kDI + c;
            red_add_v2(dst, v[hf][2 * e], v[hf][2 * e + 1]);
            red_add_v2(dst + 8, v[hf][4 + 2 * e], v[hf][4 + 2 * e + 1]);
          }
        }
      return true;
    };
    for (int k = blockIdx.x; k < total; k += gridDim.x) {
      klb::Block bk;
      if (!klb::block_of<kQB, kTK>(cu, cu_cmp, B, r, total, k, bk, pos0) || bk.ntiles == 0) continue;
      // the block's normalisers and gates (rows past the block's end read as masked)
      if (tid < kQB * kNH) {
        const int qq = tid / kNH, h = tid % kNH;
        const float L = qq < bk.nq ? teacher_lse[(int64_t)(bk.seq0 + bk.q0 + qq) * kNH + h] : -INFINITY;
        s_L[qq][h] = isfinite(L) ? -L * kLog2e : 0.f;
      } else if (tid < kQB * kNH + kQB * kHI) {
        const int i = tid - kQB * kNH, qq = i / kHI, h = i % kHI;
        s_w[qq][h] = qq < bk.nq ? __bfloat162float(w[(int64_t)(bk.seq0 + bk.q0 + qq) * kHI + h]) : 0.f;
      } else if (tid < kQB * kNH + kQB * kHI + kQB) {
        const int qq = tid - kQB * kNH - kQB * kHI;
        s_lseI[qq] = qq < bk.nq ? student_lse[bk.seq0 + bk.q0 + qq] : -INFINITY;
      }
      named_sync(1, kComputeThreads);
      const int nvis_q = (bk.q0 + q + bk.p0 + 1) / r;
      const bool q_ok = q < bk.nq && isfinite(s_lseI[q]);
      const float lseI = s_lseI[q];
      const int rot = ((bk.q0 + bk.p0) / kQB) % bk.ntiles;  // by position: results do not depend on the packing
      float dwa[kHI];
#pragma unroll
      for (int h = 0; h < kHI; ++h) dwa[h] = 0.f;
      bool fail = false;
      int64_t prev_row0 = 0;
      int prev_nvalid = 0;
      for (int ii = 0; ii < bk.ntiles; ++ii, ++t) {
        const int tj = rotated_tile(ii, rot, bk.ntiles) * kTK;
        const int j = tj + rowl;  // entry index within the sequence
        bool okw = mbar_wait_bounded(bar_sfull, t & 1u, status);
        if (__any_sync(0xffffffffu, !okw)) { fail = true; break; }
        tc::fence_after_sync();
        // the scores in two 32-head halves (the second read before the first is
        // used would need 64 registers per thread)
        uint32_t ri[kHI];
        uint32_t xs[32];
        tc::tmem_ld8_sync(tmem + lane_off + kColI + q * kHI, ri);
        tc::tmem_ld32_sync(tmem + lane_off + kColS + q * kNH, xs);
        const bool live = q_ok && j < nvis_q;
        const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
        uint64_t pa = f2_pack(0.f, 0.f), pb = pa;
        const float4* L4 = reinterpret_cast<const float4*>(&s_L[q][0]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (hh == 1) {
            tc::tmem_ld32_sync(tmem + lane_off + kColS + q * kNH + 32, xs);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sfree);
          }
          if (live) {
            // teacher p(j): the mean over heads of exp2(s scale log2e - lse_h log2e)
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
              const float4 L = L4[hh * 8 + h4];
              float a0, a1, a2, a3;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(xs[4 * h4 + 0]), __uint_as_float(xs[4 * h4 + 1])), sc2,
                               f2_pack(L.x, L.y)), a0, a1);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(xs[4 * h4 + 2]), __uint_as_float(xs[4 * h4 + 3])), sc2,
                               f2_pack(L.z, L.w)), a2, a3);
              pa = f2_add(pa, f2_pack(ex2(a0), ex2(a1)));
              pb = f2_add(pb, f2_pack(ex2(a2), ex2(a3)));
            }
          }
        }
        float g = 0.f;
        if (live) {
          float p0, p1, p2, p3;
          f2_unpack(pa, p0, p1);
          f2_unpack(pb, p2, p3);
          const float p = ((p0 + p1) + (p2 + p3)) * (1.f / kNH);
          float iv = 0.f;
#pragma unroll
          for (int h = 0; h < kHI; ++h) iv = fmaf(s_w[q][h], fmaxf(__uint_as_float(ri[h]), 0.f), iv);
          g = grad_scale * (__expf(iv - lseI) - p);
        }
        // dw partials and this entry's row of C^T (bf16, the block's 32 columns)
        uint32_t cp[kHI / 2];
#pragma unroll
        for (int h = 0; h < kHI; h += 2) {
          const float a0 = __uint_as_float(ri[h]), a1 = __uint_as_float(ri[h + 1]);
          dwa[h] = fmaf(g, fmaxf(a0, 0.f), dwa[h]);
          dwa[h + 1] = fmaf(g, fmaxf(a1, 0.f), dwa[h + 1]);
          cp[h / 2] = pack_bf16x2(a0 > 0.f ? g * s_w[q][h] : 0.f, a1 > 0.f ? g * s_w[q][h + 1] : 0.f);
        }
        if (t > 0) {  // the previous tile's products have read the C^T tile
          okw = mbar_wait_bounded(bar_cfree, (t - 1) & 1u, status);
          if (__any_sync(0xffffffffu, !okw)) { fail = true; break; }
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(base + kCOff + tc::sw128_offset(rowl, q)),
                     "r"(cp[0]), "r"(cp[1]), "r"(cp[2]), "r"(cp[3])
                     : "memory");
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cfull);
        if (ii > 0 && !epilogue(t - 1, prev_row0, prev_nvalid)) { fail = true; break; }
        prev_row0 = (int64_t)bk.cmp0 + tj;
        prev_nvalid = bk.nvis_max - tj;
      }
      if (!fail && !epilogue(t - 1, prev_row0, prev_nvalid)) fail = true;
      // dw: the per-entry partials summed over the warpgroup's 128 threads
#pragma unroll
      for (int h = 0; h < kHI; ++h) {
        float v = dwa[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_dw[warp][h] = v;
      }
      // dqI: dqI^T lanes 0..63 (dims) x columns (query, head), read by warps 0 and 1
      if (!fail && warp < 2) {
        const bool okd = mbar_wait_bounded(bar_dqdone, nblk & 1u, status);
        if (__any_sync(0xffffffffu, !okd)) {
          fail = true;
        } else {
          tc::fence_after_sync();
          uint32_t v[32];
          tc::tmem_ld32_sync(tmem + lane_off + kColDQ, v);
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dqfree);
          const int dim = rowl;
#pragma unroll
          for (int c = 0; c < kQB * kHI; ++c) {
            const int qq = c / kHI, h = c % kHI;
            if (qq < bk.nq)
              dqI[((int64_t)(bk.seq0 + bk.q0 + qq) * kHI + h) * kDI + dim] = __float2bfloat16_rn(__uint_as_float(v[c]));
          }
        }
      }
      if (fail) *abort_flag = 1;
      ++nblk;
      named_sync(1, kComputeThreads);
      if (tid < kQB * kHI) {
        const int qq = tid / kHI, h = tid % kHI;
        if (qq < bk.nq) {
          const float v = (s_dw[qq * 4][h] + s_dw[qq * 4 + 1][h]) + (s_dw[qq * 4 + 2][h] + s_dw[qq * 4 + 3][h]);
          dw[(int64_t)(bk.seq0 + bk.q0 + qq) * kHI + h] = __float2bfloat16_rn(v);
        }
      }
      named_sync(1, kComputeThreads);
      if (*abort_flag) break;  // uniform: read after the barrier
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

bool indexer_kl_bwd_tc_supported(const KLBwdArgs& a, bool fp32) {
  return !fp32 && a.idx == nullptr && a.lse_cmp != nullptr && a.student_lse != nullptr && a.H == kNH &&
         a.d == kDim && a.H_I == kHI && a.d_I == kDI;
}

cudaError_t launch_indexer_kl_bwd_tc(const KLBwdArgs& a, cudaStream_t stream) {
  if (a.T_cap <= 0) return cudaSuccess;
  const uint64_t n_cmp_rows = (uint64_t)(a.n_cmp_cap > 0 ? a.n_cmp_cap : 1);
  CUtensorMap mq, mk, mqi, mki;
  if (!make_tmap_bf16_sw128(&mq, a.q, (uint64_t)a.T_cap * kNH, kDim, 128) ||
      !make_tmap_bf16_sw128(&mk, a.k_cmp, n_cmp_rows, kDim, kTK) ||
      !make_tmap_bf16_sw128(&mqi, a.qI, (uint64_t)a.T_cap * kHI, kDI, kQB * kHI) ||
      !make_tmap_bf16_sw128(&mki, a.kI, n_cmp_rows, kDI, kTK))
    return cudaErrorInvalidValue;
  // rows without visible entries (and capacity rows) keep zero gradients
  cudaError_t err = cudaMemsetAsync(a.dkI, 0, (size_t)a.n_cmp_cap * kDI * 4, stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(a.dqI, 0, (size_t)a.T_cap * kHI * kDI * 2, stream);
  if (err == cudaSuccess) err = cudaMemsetAsync(a.dw, 0, (size_t)a.T_cap * kHI * 2, stream);
  if (err != cudaSuccess) return err;
  const size_t smem = kSmemBytes + 1024;
  err = cudaFuncSetAttribute(indexer_kl_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int blocks = (a.T_cap + kQB - 1) / kQB + a.B;  // upper bound on query blocks
  const int grid = blocks < sms ? blocks : sms;
  constexpr float kLog2e = 1.4426950408889634f;
  indexer_kl_bwd_tc_kernel<<<grid, kThreads, smem, stream>>>(
      mq, mk, mqi, mki, static_cast<const __nv_bfloat16*>(a.w), a.lse_cmp, a.student_lse, a.cu, a.cu_cmp, a.B, a.r,
      a.scale * kLog2e, a.grad_scale, static_cast<__nv_bfloat16*>(a.dqI), static_cast<__nv_bfloat16*>(a.dw), a.dkI,
      a.status, a.pos0);
  return cudaGetLastError();
}

}  // namespace csa
