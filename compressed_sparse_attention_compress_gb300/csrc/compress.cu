// compress.cu -- learned-score block compression of KV / indexer-K rows.
//
// "DeepSeek-V4 Attention Training Systems": §4 (only complete groups are
// compressed; compression resets at packed-sample boundaries), §5.1 (spans
// D_compress = 8 for overlapping ratio-4 CSA, 128 for ratio-128 HCA), §8.2
// ("C4/C128 compression": learned-score reduction), §9 (FP32 positional
// parameter, FP32 math).
//
// One CTA owns a run of consecutive entries of one sequence.  The raw rows the
// run needs are one contiguous span of the packed x and z arrays, so a single
// thread stages both spans into shared memory with bulk asynchronous copies
// (cp.async.bulk, completion on an mbarrier); every input byte is read from
// HBM once per CTA and the overlap between neighbouring entries is served from
// shared memory.  Threads then walk (entry, channel) pairs with a one-pass
// online softmax over the span in float32 and store coalesced rows.
#include "common.cuh"
#include "launch.h"

namespace csa {

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256)
compress_kernel(const TIn* __restrict__ x, const TIn* __restrict__ z, const float* __restrict__ P,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_cmp, int B, int D,
                int r, int S, int E, int rows_max, TOut* __restrict__ out, int* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_b, s_j0, s_j1;

  if (threadIdx.x == 0) {
    // blockIdx.x counts chunks of E entries over the sequences in order.
    int c = blockIdx.x, b = -1, n = 0;
    for (int bb = 0; bb < B; ++bb) {
      int L = __ldg(cu + bb + 1) - __ldg(cu + bb);
      if (L < 0) { raise_status(status, CSA_ERR_DEVICE_BOUNDS); L = 0; }
      n = L / r;
      const int nch = (n + E - 1) / E;
      if (c < nch) { b = bb; break; }
      c -= nch;
    }
    s_b = b;
    s_j0 = c * E;
    s_j1 = b >= 0 ? min(c * E + E, n) : 0;
  }
  __syncthreads();
  const int b = s_b;
  if (b < 0) return;
  const int j0 = s_j0, j1 = s_j1;
  const int tok0 = max(0, r * j0 + r - S);  // first local token the run reads
  const int tok1 = r * j1;                  // one past the last
  const int R = tok1 - tok0;                // <= rows_max by construction of E
  const int64_t row0 = (int64_t)__ldg(cu + b) + tok0;
  TIn* sx = reinterpret_cast<TIn*>(smem);
  TIn* sz = sx + (size_t)rows_max * D;
  const uint32_t bar_a = smem_u32(&bar);

  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)R * D * sizeof(TIn);
    mbar_arrive_expect_tx(bar_a, 2u * bytes);
    constexpr uint32_t kPiece = 32768;
    const char* gx = reinterpret_cast<const char*>(x + row0 * D);
    const char* gz = reinterpret_cast<const char*>(z + row0 * D);
    for (uint32_t off = 0; off < bytes; off += kPiece) {
      const uint32_t len = min(kPiece, bytes - off);
      bulk_g2s(smem_u32(sx) + off, gx + off, len, bar_a);
      bulk_g2s(smem_u32(sz) + off, gz + off, len, bar_a);
    }
  }
  if (!mbar_wait_bounded(bar_a, 0, status)) return;

  const int64_t out0 = (int64_t)__ldg(cu_cmp + b);
  const int work = (j1 - j0) * D;
  for (int i = threadIdx.x; i < work; i += blockDim.x) {
    const int e = i / D, c = i - e * D;
    const int j = j0 + e;
    const int first = r * j + r - S;
    float m = -INFINITY, den = 0.f, num = 0.f;
    for (int u = max(0, -first); u < S; ++u) {
      const int srow = first + u - tok0;
      const float lg = to_f32(sz[(size_t)srow * D + c]) + __ldg(P + (size_t)u * D + c);
      const float xv = to_f32(sx[(size_t)srow * D + c]);
      if (lg > m) {
        const float sc = expf(m - lg);
        den *= sc;
        num *= sc;
        m = lg;
      }
      const float ex = expf(lg - m);
      den += ex;
      num = fmaf(ex, xv, num);
    }
    out[(out0 + j) * D + c] = from_f32<TOut>(num / den);
  }
}

// Rows of the staging buffer and entries per CTA for a given span.
static void compress_plan(int D, int r, int S, int in_bytes, int* rows_max, int* E, size_t* smem) {
  int rows = S > 128 ? S : 128;
  if ((size_t)2 * rows * D * in_bytes > 200 * 1024) rows = S;
  *rows_max = rows;
  *E = (rows - (S - r)) / r;
  *smem = (size_t)2 * rows * D * in_bytes;
}

bool compress_supported(int D, int r, int S, int in_bytes) {
  int rows, E;
  size_t smem;
  compress_plan(D, r, S, in_bytes, &rows, &E, &smem);
  return E >= 1 && smem <= 200 * 1024;
}

template <typename TIn, typename TOut>
static cudaError_t launch_compress_t(const void* x, const void* z, const float* P, const int32_t* cu,
                                     const int32_t* cu_cmp, int B, int T_cap, int D, int r, int S,
                                     void* out, int* status, cudaStream_t stream) {
  int rows_max, E;
  size_t smem;
  compress_plan(D, r, S, (int)sizeof(TIn), &rows_max, &E, &smem);
  auto kern = compress_kernel<TIn, TOut>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long chunks = (long long)T_cap / ((long long)r * E) + B + 1;
  if (chunks <= 0) return cudaSuccess;
  kern<<<(unsigned)chunks, 256, smem, stream>>>(static_cast<const TIn*>(x), static_cast<const TIn*>(z), P,
                                                cu, cu_cmp, B, D, r, S, E, rows_max,
                                                static_cast<TOut*>(out), status);
  return cudaGetLastError();
}

cudaError_t launch_compress(const void* x, const void* z, const float* P, const int32_t* cu,
                            const int32_t* cu_cmp, int B, int T_cap, int D, int r, int S, bool fp32,
                            void* out, int* status, cudaStream_t stream) {
  if (fp32)
    return launch_compress_t<float, float>(x, z, P, cu, cu_cmp, B, T_cap, D, r, S, out, status, stream);
  return launch_compress_t<__nv_bfloat16, __nv_bfloat16>(x, z, P, cu, cu_cmp, B, T_cap, D, r, S, out,
                                                         status, stream);
}

// cu_cmp[b] = sum_{b'<b} floor(L_b' / r); also checks cu_seqlens.
__global__ void compressed_offsets_kernel(const int32_t* __restrict__ cu, int B, int r,
                                          int32_t* __restrict__ cu_cmp, int* status) {
  // one warp; B is small (one entry per packed sequence)
  const int lane = threadIdx.x;
  int carry = 0;
  if (lane == 0) cu_cmp[0] = 0;
  if (lane == 0 && __ldg(cu) != 0) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
  for (int base = 0; base < B; base += 32) {
    const int b = base + lane;
    int n = 0;
    if (b < B) {
      int L = __ldg(cu + b + 1) - __ldg(cu + b);
      if (L < 0) { raise_status(status, CSA_ERR_DEVICE_BOUNDS); L = 0; }
      n = r > 0 ? L / r : 0;
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (b < B) cu_cmp[b + 1] = carry + incl;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
}

cudaError_t launch_compressed_offsets(const int32_t* cu, int B, int r, int32_t* cu_cmp, int* status,
                                      cudaStream_t stream) {
  compressed_offsets_kernel<<<1, 32, 0, stream>>>(cu, B, r, cu_cmp, status);
  return cudaGetLastError();
}

}  // namespace csa
