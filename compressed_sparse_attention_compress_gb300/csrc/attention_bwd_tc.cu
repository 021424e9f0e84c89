// attention_bwd_tc.cu -- attention backward on tcgen05 tensor cores, 64 heads x
// 128 dims, one shared K = V head (bf16): dq and the shared-KV gradient from the
// saved output and LSE.
//
// "DeepSeek-V4 Attention Training Systems": §8.2 (the main attention backward
// consumes the saved output/LSE and produces Q, KV and attention-sink gradients
// without materializing a dense attention matrix), §9 (FP32 softmax math).
//
// Tiles are transposed as in the forward: the 128 gathered keys are the M
// dimension.  Per tile, with scale*dS = scale P (dP - D):
//   S^T[key, h]   = K[key, :] . Q[h, :]          (M=128, N=64,  K=128 dims)
//   dP^T[key, h]  = K[key, :] . dO[h, :]         (M=128, N=64,  K=128 dims; V = K)
//   dQ^T[dim, h] += K^T[dim, key] dS^T[key, h]   (M=128, N=64,  K=128 keys)
//   dKV[key, dim] = dS^T[key, h] Q[h, dim] + P^T[key, h] dO[h, dim]
//                                                (M=128, N=128, K=64 heads, twice)
// The bf16 P^T and dS^T tiles are written once by the softmax warps and read
// twice: as the MN-major B operand of dQ^T and as the K-major A operand of
// dKV (the same 128-byte-swizzled rows); Q and dO likewise serve as K-major B
// of S^T / dP^T and MN-major B of dKV.  Tensor memory: S^T 64, dP^T 64, dQ^T
// 64 and two 128-column dKV buffers (448 of 512 columns).
//
// Warp roles, one query stream per CTA (one CTA per SM, persistent):
//   producer (1 warp): the forward's gather -- index list read a tile ahead,
//     empty compressed tiles skipped, rows copied with coalesced 16-byte
//     cp.async into a 2-stage ring; Q and dO of each query;
//   MMA issuer (1 warp): S^T and dP^T of a tile as soon as it is gathered and
//     the previous scores are read; dQ^T and dKV once P^T / dS^T are written;
//   softmax (8 warps, thread = (key, 32 heads)): P = exp2(S scale log2e - lse),
//     scale dS, the two bf16 tiles; at the end of a query dQ^T -> dq;
//   epilogue (4 warps): each dKV tile added to the float32 gradient rows with
//     red.global.add.v2, four threads per 32-byte row piece (the 16x256b
//     tensor-memory read), while the next tile is computed.
// Every wait is bounded (CSA_ERR_DEVICE_TIMEOUT and a uniform abort).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "ws_sync.cuh"

namespace csa {

namespace {

using namespace ws;

constexpr int kTK = 128, kNH = 64, kDim = 128;
constexpr int kSoftWarps = 8, kEpiWarps = 4;
constexpr int kEpiWarp0 = kSoftWarps;                  // warps 8..11
constexpr int kProdWarp = kEpiWarp0 + kEpiWarps;       // warp 12
constexpr int kMmaWarp = kProdWarp + 1;                // warp 13
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kRowsPerLane = kTK / 32;                 // producer rows per lane
constexpr int kStages = 4;                             // key-tile ring

constexpr uint32_t kQRegion = kNH * 128;               // 8 KB: 64 rows x 64 dims
constexpr uint32_t kQBytes = 2 * kQRegion;             // 16 KB
constexpr uint32_t kTileRegion = kTK * 128;            // 16 KB
constexpr uint32_t kTileBytes = 2 * kTileRegion;       // 32 KB
constexpr uint32_t kQOff = 0;
constexpr uint32_t kGOff = kQBytes;                    // dO
constexpr uint32_t kStageOff = 2 * kQBytes;            // kStages stages
constexpr uint32_t kPOff = kStageOff + kStages * kTileBytes;  // P^T [key][head]
constexpr uint32_t kDSOff = kPOff + kTK * 128;         // scale dS^T [key][head]
constexpr uint32_t kSmem = kDSOff + kTK * 128;         // 192 KB

constexpr uint32_t kColS = 0, kColDP = 64, kColDQ = 128, kColKV = 256;

enum : int { kFirst = 1, kLast = 2, kDone = 8, kCmp = 16 };

struct Meta {
  int row;
  int flags;
};

__device__ __forceinline__ void red_add_v2(float* p, uint32_t a, uint32_t b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};\n" ::"l"(p), "f"(__uint_as_float(a)), "f"(__uint_as_float(b))
               : "memory");
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
attention_bwd_tc_kernel(int kind, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cmp,
                        const __nv_bfloat16* __restrict__ k_raw, const int32_t* __restrict__ idx, int k_pad,
                        const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_cmp, int B, int T_cap, int r,
                        int window, float scale, float scale_log2, const float* __restrict__ lse,
                        const float* __restrict__ delta, const __nv_bfloat16* __restrict__ dout,
                        __nv_bfloat16* __restrict__ dq, float* __restrict__ dkv_cmp, float* __restrict__ dkv_raw,
                        int* status,
                        const int32_t* __restrict__ pos0) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages], s_kvfull[2], s_kvfree[2];
  __shared__ __align__(8) uint64_t s_qfull, s_qempty, s_sfull, s_sfree, s_pfull, s_pfree, s_dqdone, s_dqfree;
  __shared__ __align__(8) uint64_t s_drain;  // the MMA thread's last commit, before tensor memory is freed
  __shared__ Meta s_meta[kStages];
  __shared__ int s_rows[kStages][kTK];
  __shared__ float s_lse2[kNH], s_D[kNH];
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = smem_u32(&s_full[0]), bar_empty = smem_u32(&s_empty[0]);
  const uint32_t bar_kvfull = smem_u32(&s_kvfull[0]), bar_kvfree = smem_u32(&s_kvfree[0]);

  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_u32(&s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 64);        // 32 cp.async arrivals + the warp's release
      mbar_init(bar_empty + 8 * s, 1 + kEpiWarps);  // MMA done with the tile + each epilogue warp done with its rows
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_kvfull + 8 * s, 1);
      mbar_init(bar_kvfree + 8 * s, kEpiWarps);
    }
    mbar_init(smem_u32(&s_qfull), 64);
    mbar_init(smem_u32(&s_qempty), 1);
    mbar_init(smem_u32(&s_sfull), 1);
    mbar_init(smem_u32(&s_sfree), kSoftWarps);
    mbar_init(smem_u32(&s_pfull), kSoftWarps);
    mbar_init(smem_u32(&s_pfree), 1);
    mbar_init(smem_u32(&s_dqdone), 1);
    mbar_init(smem_u32(&s_dqfree), kSoftWarps);
    mbar_init(smem_u32(&s_drain), 1);
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

  if (warp == kProdWarp) {
    // =================== producer: lane pt owns rows pt + 32 i of every tile ===================
    const int pt = lane;
    uint32_t n = 0, nq = 0;  // tiles and queries produced
    bool alive = true;
    for (int ord = 0; alive; ++ord) {
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
      int pre[kRowsPerLane];
#pragma unroll
      for (int i = 0; i < kRowsPerLane; ++i) pre[i] = -1;
      auto prefetch = [&](int it) {
        if (kind == kAttnCSA && it < nct) {
          const int32_t* src = idx + (int64_t)row * k_pad;
#pragma unroll
          for (int i = 0; i < kRowsPerLane; ++i) {
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
        int rr[kRowsPerLane];
        bool any = false;
#pragma unroll
        for (int i = 0; i < kRowsPerLane; ++i) {
          rr[i] = resolve(it, pt + 32 * i, pre[i]);
          any = any || rr[i] >= 0;
        }
        prefetch(it + 1);
        if (it < nct && !__any_sync(0xffffffffu, any)) continue;  // empty compressed tile
        const uint32_t st = n % kStages;
        bool ok = mbar_wait_bounded(bar_empty + 8 * st, ((n / kStages) & 1u) ^ 1u, status);
        if (first && nq > 0) ok = ok && mbar_wait_bounded(smem_u32(&s_qempty), (nq - 1) & 1u, status);
        if (__any_sync(0xffffffffu, !ok || *abort_flag != 0)) {
          *abort_flag = 1;
          alive = false;
          break;
        }
        if (first) {  // this query's Q and dO (64 heads x 128 dims each, swizzled K-major)
#pragma unroll 4
          for (int i = pt; i < kNH * 16; i += 32) {
            const int h = i >> 4, c = i & 15;
            const uint32_t off = (c >> 3) * kQRegion + tc::sw128_offset(h, c & 7);
            cp_async_16(base + kQOff + off, q + ((int64_t)row * kNH + h) * kDim + c * 8);
            cp_async_16(base + kGOff + off, dout + ((int64_t)row * kNH + h) * kDim + c * 8);
          }
          arrive_cp_async(smem_u32(&s_qfull));
          __syncwarp();
          if (lane == 0) arrive_warp(smem_u32(&s_qfull));
          ++nq;
        }
        const bool cmpt = it < nct;
        const __nv_bfloat16* ks = cmpt ? k_cmp : k_raw;
        const uint32_t kb = base + kStageOff + st * kTileBytes;
#pragma unroll
        for (int i = 0; i < kRowsPerLane; ++i) s_rows[st][pt + 32 * i] = rr[i];
        // coalesced gather: eight lanes per 256-byte row, four rows per step
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
        // the last tile is a window tile (the window holds the query itself), never skipped
        if (pt == 0) s_meta[st] = Meta{row, (first ? kFirst : 0) | (cmpt ? kCmp : 0) | (it == ntl - 1 ? kLast : 0)};
        arrive_cp_async(bar_full + 8 * st);
        __syncwarp();
        if (lane == 0) arrive_warp(bar_full + 8 * st);  // release: publishes s_rows / s_meta
        first = false;
        ++n;
      }
    }
    if (alive) {  // end-of-stream marker
      const uint32_t st = n % kStages;
      const bool ok = mbar_wait_bounded(bar_empty + 8 * st, ((n / kStages) & 1u) ^ 1u, status);
      if (__any_sync(0xffffffffu, !ok)) {
        *abort_flag = 1;
      } else {
        if (pt == 0) s_meta[st] = Meta{-1, kDone};
        mbar_arrive(bar_full + 8 * st);
        __syncwarp();
        if (lane == 0) arrive_warp(bar_full + 8 * st);
      }
    }
    cp_async_wait<0>();
  }
  else if (warp == kMmaWarp) {
    // =================== MMA issuer: backward products first, then the next scores ===================
    if (lane == 0) {
      constexpr uint32_t kIdQK = tc::idesc_bf16(kTK, kNH, 0, 0);   // S^T, dP^T
      constexpr uint32_t kIdDQ = tc::idesc_bf16(kDim, kNH, 1, 1);  // dQ^T += K^T dS^T
      constexpr uint32_t kIdKV = tc::idesc_bf16(kTK, kDim, 0, 1);  // dKV = dS^T Q + P^T dO
      // descriptors of K-step 0; a K-step adds its byte offset / 16 to the address field
      const uint64_t dq_b = tc::smem_desc_sw128(base + kQOff, 16, 1024);             // Q, K-major B
      const uint64_t dg_b = tc::smem_desc_sw128(base + kGOff, 16, 1024);             // dO, K-major B
      const uint64_t dk0 = tc::smem_desc_sw128(base + kStageOff, 16, 1024);          // K tile, K-major A
      const uint64_t dkt0 = tc::smem_desc_sw128(base + kStageOff, kTileRegion, 1024);  // K tile as K^T, MN-major A
      const uint64_t dds_b = tc::smem_desc_sw128(base + kDSOff, 1024, 1024);         // dS^T, MN-major B
      const uint64_t dds_a = tc::smem_desc_sw128(base + kDSOff, 16, 1024);           // dS^T, K-major A
      const uint64_t dp_a = tc::smem_desc_sw128(base + kPOff, 16, 1024);             // P^T, K-major A
      const uint64_t dq_mn = tc::smem_desc_sw128(base + kQOff, kQRegion, 1024);      // Q, MN-major B
      const uint64_t dg_mn = tc::smem_desc_sw128(base + kGOff, kQRegion, 1024);      // dO, MN-major B
      constexpr uint64_t kStageStep = kTileBytes >> 4;
      const uint32_t pfull = smem_u32(&s_pfull), sfree = smem_u32(&s_sfree), dqfree = smem_u32(&s_dqfree);
      uint32_t kq = 0, kp = 0, nqq = 0, nqp = 0;  // score / backward tiles issued, queries started by each
      bool end = false;                           // the end-of-stream tile was seen
      uint64_t last = globaltimer_ns();
      while (!(end && kp == kq)) {
        bool progress = false;
        if (kp < kq && mbar_test(pfull, kp & 1u)) {
          const uint32_t sp = kp % kStages;      // stage of tile kp
          const uint32_t bkv = kp & 1u;          // its dKV buffer
          const int flags = s_meta[sp].flags;
          const bool first = (flags & kFirst) != 0;
          const bool kv_ok = kp < 2 || mbar_test(bar_kvfree + 8 * bkv, ((kp >> 1) - 1) & 1u);
          const bool dq_ok = !first || nqp == 0 || mbar_test(dqfree, (nqp - 1) & 1u);
          if (kv_ok && dq_ok) {
            if (first) ++nqp;
            tc::fence_after_sync();
            const uint64_t dkt = dkt0 + sp * kStageStep;
#pragma unroll
            for (int ks = 0; ks < kTK / 16; ++ks) {  // dQ^T over the tile's keys, 16 at a time
              const uint32_t off = (ks * 2048) >> 4;
              tc::mma_bf16(tmem + kColDQ, dkt + off, dds_b + off, kIdDQ, (first && ks == 0) ? 0u : 1u);
            }
            const uint32_t tkv = tmem + kColKV + bkv * 128;
#pragma unroll
            for (int kh = 0; kh < kNH / 16; ++kh)    // dS^T Q over the heads, 16 at a time
              tc::mma_bf16(tkv, dds_a + ((kh * 32) >> 4), dq_mn + ((kh * 2048) >> 4), kIdKV, kh > 0 ? 1u : 0u);
#pragma unroll
            for (int kh = 0; kh < kNH / 16; ++kh)    // + P^T dO
              tc::mma_bf16(tkv, dp_a + ((kh * 32) >> 4), dg_mn + ((kh * 2048) >> 4), kIdKV, 1u);
            tc::mma_commit(smem_u32(&s_pfree));
            tc::mma_commit(bar_kvfull + 8 * bkv);
            tc::mma_commit(bar_empty + 8 * sp);
            if (flags & kLast) {
              tc::mma_commit(smem_u32(&s_dqdone));
              tc::mma_commit(smem_u32(&s_qempty));
            }
            ++kp;
            progress = true;
          }
        }
        if (!end && kq < kp + 2 && mbar_test(bar_full + 8 * (kq % kStages), (kq / kStages) & 1u)) {
          const uint32_t st = kq % kStages;
          const int flags = s_meta[st].flags;
          if (flags & kDone) {
            end = true;
            progress = true;
          } else if ((kq == 0 || mbar_test(sfree, (kq - 1) & 1u)) &&
                     (!(flags & kFirst) || mbar_test(smem_u32(&s_qfull), nqq & 1u))) {
            if (flags & kFirst) ++nqq;
            tc::fence_after_sync();
            const uint64_t dk = dk0 + st * kStageStep;
#pragma unroll
            for (int ks = 0; ks < kDim / 16; ++ks) {
              const uint32_t off = ((ks >> 2) * kTileRegion + (ks & 3) * 32) >> 4;
              const uint32_t offq = ((ks >> 2) * kQRegion + (ks & 3) * 32) >> 4;
              tc::mma_bf16(tmem + kColS, dk + off, dq_b + offq, kIdQK, ks > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int ks = 0; ks < kDim / 16; ++ks) {
              const uint32_t off = ((ks >> 2) * kTileRegion + (ks & 3) * 32) >> 4;
              const uint32_t offq = ((ks >> 2) * kQRegion + (ks & 3) * 32) >> 4;
              tc::mma_bf16(tmem + kColDP, dk + off, dg_b + offq, kIdQK, ks > 0 ? 1u : 0u);
            }
            tc::mma_commit(smem_u32(&s_sfull));
            ++kq;
            progress = true;
          }
        }
        if (progress) {
          last = globaltimer_ns();
        } else {
          if (*abort_flag) break;
          if (globaltimer_ns() - last > kWaitLimitNs) {
            raise_status(status, CSA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          if (kp < kq) mbar_sleep(pfull, kp & 1u, 500);
          else if (!end) mbar_sleep(bar_full + 8 * (kq % kStages), (kq / kStages) & 1u, 500);
          else __nanosleep(64);
        }
      }
      // every MMA this thread issued has completed before tensor memory is freed (also after an abort)
      tc::mma_commit(smem_u32(&s_drain));
      mbar_wait_bounded(smem_u32(&s_drain), 0, status);
    }
  } else if (warp < kSoftWarps) {
    // =================== softmax: warp = (head half, lane quadrant), thread = (key, 32 heads) ===================
    const int quad = warp & 3, hh = warp >> 2;
    const int key = quad * 32 + lane;            // tensor-memory lane: key of the tile / head dim
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + kColS + hh * 32;
    const uint32_t t_dp = tmem + lane_off + kColDP + hh * 32;
    const uint32_t t_dq = tmem + lane_off + kColDQ + hh * 32;
    constexpr int kBar = 1;
    constexpr float kLog2e = 1.4426950408889634f;
    const uint32_t prow = base + kPOff, dsrow = base + kDSOff;
    uint32_t k = 0, nq = 0;
    int row = -1;
    for (uint32_t n = 0;; ++n) {
      const uint32_t st = n % kStages;
      const bool okf = mbar_wait_bounded(bar_full + 8 * st, (n / kStages) & 1u, status);
      if (bar_or(kBar, kSoftThreads, !okf || *abort_flag != 0)) {
        *abort_flag = 1;
        break;
      }
      const Meta mt = s_meta[st];
      if (mt.flags & kDone) break;
      if (mt.flags & kFirst) {  // this query's per-head lse (log2 units) and D = dout . out
        row = mt.row;
        bar_sync(kBar, kSoftThreads);
        if (tid < kNH) {
          s_lse2[tid] = __ldg(lse + (int64_t)row * kNH + tid) * kLog2e;
          s_D[tid] = __ldg(delta + (int64_t)row * kNH + tid);
        }
        bar_sync(kBar, kSoftThreads);
      }
      const bool valid = s_rows[st][key] >= 0;
      bool ok = mbar_wait_bounded(smem_u32(&s_sfull), k & 1u, status);
      tc::fence_after_sync();
      uint32_t rs[32], rd[32];
      tc::tmem_ld32_sync(t_s, rs);
      tc::tmem_ld32_sync(t_dp, rd);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_sfree));
      // P and scale * dS of this key for 32 heads, packed to bf16 pairs
      uint32_t pp[16], dd[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int h = hh * 32 + j;
        float p0 = 0.f, p1 = 0.f;
        if (valid) {
          p0 = ex2(fmaf(__uint_as_float(rs[j]), scale_log2, -s_lse2[h]));
          p1 = ex2(fmaf(__uint_as_float(rs[j + 1]), scale_log2, -s_lse2[h + 1]));
        }
        const float g0 = p0 * (__uint_as_float(rd[j]) - s_D[h]) * scale;
        const float g1 = p1 * (__uint_as_float(rd[j + 1]) - s_D[h + 1]) * scale;
        pp[j >> 1] = pack_bf16x2(p0, p1);
        dd[j >> 1] = pack_bf16x2(g0, g1);
      }
      // the previous tile's products must be done reading P^T / dS^T
      if (k > 0) ok = ok && mbar_wait_bounded(smem_u32(&s_pfree), (k - 1) & 1u, status);
      if (bar_or(kBar, kSoftThreads, !ok)) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + tc::sw128_offset(key, hh * 4 + c)),
                     "r"(pp[4 * c]), "r"(pp[4 * c + 1]), "r"(pp[4 * c + 2]), "r"(pp[4 * c + 3]));
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(dsrow + tc::sw128_offset(key, hh * 4 + c)),
                     "r"(dd[4 * c]), "r"(dd[4 * c + 1]), "r"(dd[4 * c + 2]), "r"(dd[4 * c + 3]));
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_pfull));
      ++k;
      if (mt.flags & kLast) {  // end of the query: dQ^T -> dq (this thread: head dim `key`, 32 heads)
        ok = mbar_wait_bounded(smem_u32(&s_dqdone), nq & 1u, status);
        if (bar_or(kBar, kSoftThreads, !ok)) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after_sync();
        uint32_t ro[32];
        tc::tmem_ld32_sync(t_dq, ro);
        __nv_bfloat16* drow = dq + ((int64_t)row * kNH + hh * 32) * kDim + key;
#pragma unroll
        for (int j = 0; j < 32; ++j) drow[(int64_t)j * kDim] = __float2bfloat16(__uint_as_float(ro[j]));
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_dqfree));
        ++nq;
      }
    }
  } else if (warp >= kEpiWarp0 && warp < kProdWarp) {
    // =================== epilogue: thread = key row of the dKV tile ===================
    const int ew = warp - kEpiWarp0;             // lane quadrant (warp % 4 == ew)
    const int key = ew * 32 + lane;
    const uint32_t lane_off = (uint32_t)(ew * 32) << 16;
    for (uint32_t n = 0;; ++n) {
      const uint32_t st = n % kStages, bkv = n & 1u;
      bool ok = mbar_wait_bounded(bar_full + 8 * st, (n / kStages) & 1u, status);
      if (__any_sync(0xffffffffu, !ok || *abort_flag != 0)) {
        *abort_flag = 1;
        break;
      }
      const Meta mt = s_meta[st];
      if (mt.flags & kDone) break;
      const int rr = s_rows[st][key];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);  // the rows are read; the MMA frees the tile
      ok = mbar_wait_bounded(bar_kvfull + 8 * bkv, (n >> 1) & 1u, status);
      if (__any_sync(0xffffffffu, !ok)) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      // the warp's 32 key rows as two 16-lane halves: thread = (two keys, two
      // 8-byte column pairs per 16 columns); four threads cover 32 contiguous
      // bytes of a gradient row, so each reduction instruction fills 8 sectors
      float* dstb = (mt.flags & kCmp) ? dkv_cmp : dkv_raw;
      int rk[2][2];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 2; ++e) rk[hf][e] = __shfl_sync(0xffffffffu, rr, hf * 16 + e * 8 + (lane >> 2));
      const int cc = 2 * (lane & 3);
#pragma unroll 1
      for (int c0 = 0; c0 < kDim; c0 += 16) {
        uint32_t v[2][8];
        tc::tmem_ld16x256_pair_sync(tmem + ((uint32_t)(ew * 32) << 16) + kColKV + bkv * 128 + c0,
                                    tmem + ((uint32_t)(ew * 32 + 16) << 16) + kColKV + bkv * 128 + c0, v[0], v[1]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (rk[hf][e] >= 0) {
              float* dst = dstb + (int64_t)rk[hf][e] * kDim + c0 + cc;
              red_add_v2(dst, v[hf][2 * e], v[hf][2 * e + 1]);
              red_add_v2(dst + 8, v[hf][4 + 2 * e], v[hf][4 + 2 * e + 1]);
            }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_kvfree + 8 * bkv);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, 512);
}

// Capacity rows (>= cu[B]): zero dq.
__global__ void attention_bwd_capacity_rows_kernel(const int32_t* __restrict__ cu, int B, int T_cap,
                                                   __nv_bfloat16* __restrict__ dq) {
  const int64_t first = __ldg(cu + B);
  const int64_t n = ((int64_t)T_cap - first) * kNH * kDim;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dq[first * kNH * kDim + i] = __float2bfloat16(0.f);
}

bool attention_bwd_tc_supported(const AttnBwdArgs& a, bool fp32) {
  return !fp32 && a.H == kNH && a.d == kDim && a.v_cmp == nullptr && a.v_raw == nullptr;
}

cudaError_t launch_attention_bwd_tc(AttnKind kind, const AttnBwdArgs& a, cudaStream_t stream) {
  if (a.T_cap <= 0) return cudaSuccess;
  const size_t smem = kSmem + 1024;
  cudaError_t err =
      cudaFuncSetAttribute(attention_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  attention_bwd_capacity_rows_kernel<<<sms, 256, 0, stream>>>(a.cu, a.B, a.T_cap, static_cast<__nv_bfloat16*>(a.dq));
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int grid = a.T_cap < sms ? a.T_cap : sms;
  constexpr float kLog2e = 1.4426950408889634f;
  attention_bwd_tc_kernel<<<grid, kThreads, smem, stream>>>(
      (int)kind, static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_cmp),
      static_cast<const __nv_bfloat16*>(a.k_raw), a.idx, a.k_pad, a.cu, a.cu_cmp, a.B, a.T_cap, a.r, a.window,
      a.scale, a.scale * kLog2e, a.lse, a.delta, static_cast<const __nv_bfloat16*>(a.dout),
      static_cast<__nv_bfloat16*>(a.dq), a.dk_cmp, a.dk_raw, a.status, a.pos0);
  return cudaGetLastError();
}

}  // namespace csa
