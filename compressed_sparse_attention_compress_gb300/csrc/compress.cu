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
// shared memory.  A thread owns a pair of adjacent channels and walks the
// run's entries; per entry it takes the span in chunks of 8 positions: the
// chunk's logits z + P (log2 domain) in registers, one max, one rescale of the
// running sums, then ex2 (MUFU) weights -- a float32 softmax over the span,
// stored as a coalesced pair of the output row.
#include "common.cuh"
#include "launch.h"

namespace csa {

namespace {

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float2 load_pair(const __nv_bfloat16* p) {
  const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(bf16_lo(v), bf16_hi(v));
}
__device__ __forceinline__ float2 load_pair(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ void store_pair(__nv_bfloat16* p, float a, float b) {
  *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(a, b);
}
__device__ __forceinline__ void store_pair(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}

}  // namespace

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256)
compress_kernel(const TIn* __restrict__ x, const TIn* __restrict__ z, const float* __restrict__ P,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_cmp, int B, int D,
                int r, int S, int E, int rows_max, TOut* __restrict__ out, int* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_b, s_j0, s_j1;

  if (threadIdx.x < 32) {
    // blockIdx.x counts chunks of E entries over the sequences in order; warp 0
    // finds the owning sequence 32 sequences at a time (one load round trip each)
    const int lane = threadIdx.x;
    int c = blockIdx.x, b = -1, n = 0;
    for (int base = 0; base < B && b < 0; base += 32) {
      const int bb = base + lane;
      int L = bb < B ? __ldg(cu + bb + 1) - __ldg(cu + bb) : 0;
      if (L < 0) { raise_status(status, CSA_ERR_DEVICE_BOUNDS); L = 0; }
      const int nb = L / r;
      const int nch = (nb + E - 1) / E;
      int incl = nch;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t hit = __ballot_sync(0xffffffffu, bb < B && c < incl);
      if (hit != 0u) {
        const int w = __ffs(hit) - 1;  // first sequence whose chunks reach c
        b = base + w;
        c -= __shfl_sync(0xffffffffu, incl - nch, w);
        n = __shfl_sync(0xffffffffu, nb, w);
      } else {
        c -= __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) {
      s_b = b;
      s_j0 = c * E;
      s_j1 = b >= 0 ? min(c * E + E, n) : 0;
    }
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
  constexpr float kLog2e = 1.4426950408889634f;
  const int pairs = D >> 1;                        // D is even (checked on the host)
  const int groups = (int)blockDim.x / pairs;      // entries worked on side by side
  const int cpair = (int)threadIdx.x % pairs, eg = (int)threadIdx.x / pairs;
  if (eg >= groups) return;
  const int c = 2 * cpair;
  for (int e = eg; e < j1 - j0; e += groups) {
    const int j = j0 + e;
    const int first = r * j + r - S;               // span position u reads local token first + u
    float m0 = -INFINITY, m1 = -INFINITY, den0 = 0.f, den1 = 0.f, num0 = 0.f, num1 = 0.f;
    for (int u0 = max(0, -first); u0 < S; u0 += 8) {
      float lg0[8], lg1[8], xv0[8], xv1[8];
      float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int u = u0 + k;
        lg0[k] = -INFINITY;
        lg1[k] = -INFINITY;
        xv0[k] = 0.f;
        xv1[k] = 0.f;
        if (u < S) {
          const size_t sofs = (size_t)(first + u - tok0) * D + c;
          const float2 zz = load_pair(sz + sofs), xx = load_pair(sx + sofs);
          const float2 pp = __ldg(reinterpret_cast<const float2*>(P + (size_t)u * D + c));
          lg0[k] = (zz.x + pp.x) * kLog2e;
          lg1[k] = (zz.y + pp.y) * kLog2e;
          xv0[k] = xx.x;
          xv1[k] = xx.y;
          cm0 = fmaxf(cm0, lg0[k]);
          cm1 = fmaxf(cm1, lg1[k]);
        }
      }
      const float mn0 = fmaxf(m0, cm0), mn1 = fmaxf(m1, cm1);
      const float sc0 = ex2f(m0 - mn0), sc1 = ex2f(m1 - mn1);  // 0 while the sums are empty
      den0 *= sc0;
      num0 *= sc0;
      den1 *= sc1;
      num1 *= sc1;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float w0 = ex2f(lg0[k] - mn0), w1 = ex2f(lg1[k] - mn1);  // -inf (past the span) -> 0
        den0 += w0;
        den1 += w1;
        num0 = fmaf(w0, xv0[k], num0);
        num1 = fmaf(w1, xv1[k], num1);
      }
      m0 = mn0;
      m1 = mn1;
    }
    store_pair(out + (out0 + j) * D + c, num0 / den0, num1 / den1);
  }
}

// Rows of the staging buffer and entries per CTA for a given span.
static void compress_plan(int D, int r, int S, int in_bytes, int* rows_max, int* E, size_t* smem) {
  // runs of about 64 rows: many CTAs per SM, so one CTA's staging copy overlaps
  // another's reduction
  int rows = S > 64 ? S : 64 + (S - r);
  if ((size_t)2 * rows * D * in_bytes > 200 * 1024) rows = S;
  *rows_max = rows;
  *E = (rows - (S - r)) / r;
  *smem = (size_t)2 * rows * D * in_bytes;
}

bool compress_supported(int D, int r, int S, int in_bytes) {
  int rows, E;
  size_t smem;
  compress_plan(D, r, S, in_bytes, &rows, &E, &smem);
  // a thread takes two adjacent channels; one row of channel pairs fits the CTA
  return E >= 1 && smem <= 200 * 1024 && D % 2 == 0 && D / 2 <= 256;
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
