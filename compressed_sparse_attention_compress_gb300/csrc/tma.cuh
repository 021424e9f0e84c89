// tma.cuh -- tensor-memory-accelerator (TMA) tiled loads: host-side tensor
// map encoding for 2-D bf16 arrays with 128-byte swizzle, and the device-side
// cp.async.bulk.tensor load that completes on an mbarrier.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; no driver-library link)
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

// Encode a tensor map over a row-major bf16 array [rows, cols]: boxes of
// box_rows x 64 elements (128 bytes, the 128-byte swizzle span).  Rows past
// `rows` read as zeros.  Returns false if the driver refuses the encoding.
bool make_tmap_bf16_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// The same over a row-major 8-bit array [rows, cols] (E4M3 codes): boxes of
// box_rows x 64 bytes, 64-byte swizzle.
bool make_tmap_u8_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace csa
