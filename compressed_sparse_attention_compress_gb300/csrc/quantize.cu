// quantize.cu -- E4M3 quantisation of the indexer operands for the FP8 indexer.
//
// "DeepSeek-V4 Attention Training Systems" §1 and §9 name an FP8 indexer (FP8
// q^I / k^I for the index-search term) and fix no format.  Each row of x
// (cols <= 256) gets a power-of-two scale s = 2^e, the smallest with
// max|x| / s <= 448 -- the decision taken on max|x| / 448 in float32 -- and the
// E4M3 code of x / s, rounded to nearest even (the hardware conversion, which
// never saturates here since |x / s| <= 448).  One warp per row.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace csa {

template <typename TIn>
__global__ void __launch_bounds__(256)
quantize_fp8_kernel(const TIn* __restrict__ x, int64_t rows, int cols, uint8_t* __restrict__ codes,
                    float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const TIn* xr = x + row * cols;
  float v[8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    v[i] = c < cols ? to_f32(xr[c]) : 0.f;
    amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int e = 0;
  if (amax > 0.f) {
    int fe;
    const float fm = frexpf(__fdiv_rn(amax, 448.0f), &fe);  // ratio = fm 2^fe, fm in [0.5, 1)
    e = (fm == 0.5f) ? fe - 1 : fe;                         // smallest e with ratio <= 2^e
  }
  if (lane == 0) scales[row] = ldexpf(1.0f, e);
  const float inv = ldexpf(1.0f, -e);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    if (c < cols) codes[row * cols + c] = (uint8_t)__nv_cvt_float_to_fp8(v[i] * inv, __NV_SATFINITE, __NV_E4M3);
  }
}

cudaError_t launch_quantize_fp8(const void* x, int64_t rows, int cols, bool fp32, uint8_t* codes, float* scales,
                                cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  if (fp32)
    quantize_fp8_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), rows, cols, codes, scales);
  else
    quantize_fp8_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), rows, cols,
                                                                 codes, scales);
  return cudaGetLastError();
}

}  // namespace csa
