// tile_sm80.cuh -- gathered key tiles and the S = Q K^T warp tile shared by
// the attention and indexer-KL kernels (mma.sync m16n8k16 bf16, fp32 acc).
#pragma once

#include "common.cuh"
#include "mma_sm80.cuh"

namespace csa {

constexpr int kKeys = 64;  // keys per tile

template <int D>
struct AttnSmem {
  static constexpr int kStride = D + 8;  // bf16 elements per smem row (16 B pad)
};

// Gather one tile of key (and value) rows into shared memory.  rows[k] < 0
// leaves zeros.  bf16 sources use cp.async; float sources are converted.
// rows outside [0, row_limit) are treated like -1 (zeros), so a bad row
// number can never turn into an out-of-bounds load.
template <typename TIn, int D>
__device__ __forceinline__ void gather_tile(const TIn* __restrict__ ksrc, const TIn* __restrict__ vsrc,
                                            bool separate_v, const int* rows, int row_limit, __nv_bfloat16* sk,
                                            __nv_bfloat16* sv, int tid, int nthreads) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per bf16 row
  constexpr int kStride = AttnSmem<D>::kStride;
  for (int i = tid; i < kKeys * kChunks; i += nthreads) {
    const int k = i / kChunks, c = i - k * kChunks;
    const int row = rows[k] < row_limit ? rows[k] : -1;
    __nv_bfloat16* dk = sk + k * kStride + c * 8;
    __nv_bfloat16* dv = sv + k * kStride + c * 8;
    if constexpr (sizeof(TIn) == 2) {
      const TIn* gk = ksrc + (int64_t)(row < 0 ? 0 : row) * D + c * 8;
      cp_async_16_zfill(smem_u32(dk), gk, row >= 0);
      if (separate_v) {
        const TIn* gv = vsrc + (int64_t)(row < 0 ? 0 : row) * D + c * 8;
        cp_async_16_zfill(smem_u32(dv), gv, row >= 0);
      }
    } else {
      uint4 vk = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (row >= 0) {
        vk = Load8<TIn>::run(ksrc + (int64_t)row * D + c * 8);
        if (separate_v) vv = Load8<TIn>::run(vsrc + (int64_t)row * D + c * 8);
      }
      *reinterpret_cast<uint4*>(dk) = vk;
      if (separate_v) *reinterpret_cast<uint4*>(dv) = vv;
    }
  }
}


// s[n][e] = Q K^T for this warp's 16 query rows (sQ rows warp*16..) against
// the 64 keys of tK, in the mma.sync C layout: row lane/4 + 8*(e>>1), key
// n*8 + 2*(lane&3) + (e&1).
template <int D>
__device__ __forceinline__ void qk_tile(const __nv_bfloat16* sQ, const __nv_bfloat16* tK, int warp, int lane,
                                        float (&s)[8][4]) {
  constexpr int kStride = AttnSmem<D>::kStride;
#pragma unroll
  for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t a[4];
    ldmatrix_x4(smem_u32(sQ + (warp * 16 + (lane & 15)) * kStride + kk * 16 + (lane >> 4) * 8), a[0], a[1],
                a[2], a[3]);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t bq[4];
      const int key = np * 16 + (lane & 7) + (lane >> 4) * 8;
      const int col = kk * 16 + ((lane >> 3) & 1) * 8;
      ldmatrix_x4(smem_u32(tK + key * kStride + col), bq[0], bq[1], bq[2], bq[3]);
      mma_bf16_16816(s[2 * np], a, bq);
      mma_bf16_16816(s[2 * np + 1], a, bq + 2);
    }
  }
}

}  // namespace csa
