// compress.cu -- learned-score block compression of KV / indexer-K rows.
//
// "DeepSeek-V4 Attention Training Systems": §4 (only complete groups are
// compressed; compression resets at packed-sample boundaries), §5.1 (spans
// D_compress = 8 for overlapping ratio-4 CSA, 128 for ratio-128 HCA), §8.2
// ("C4/C128 compression": learned-score reduction), §9 (FP32 positional
// parameter, FP32 math), §10 ("compressor softmax and normalization
// intermediates"), §12 ("RoPE mode is per layer and per compressed coordinate
// system").
//
// One kernel serves csa_compress and csa_compress_ex.  A CTA owns a run of
// consecutive entries of one sequence.  The raw rows the run needs are one
// contiguous span of each packed input stream, so a single thread stages them
// into shared memory with bulk asynchronous copies (cp.async.bulk, completion
// on an mbarrier): every input byte is read from HBM once per CTA and the
// overlap between neighbouring entries is served from shared memory.
//
// One warp owns an entry (two entries per warp at D = 32): lane l takes the
// channel pairs l, l+32, ... so every shared-memory read is one coalesced row
// segment.  Per pair and span position: the logit z + P, one running maximum
// per chunk of 8 positions, ex2 (MUFU) weights of (logit - max) * log2(e) --
// a float32 softmax over the span.  The extras of csa_compress_ex follow
// before the single rounding of the output:
//   * a second (x_prev, z_prev) stream that span positions u < r (the previous
//     block of an overlapping span) read instead of (x, z);
//   * RMSNorm over the entry's D channels (a warp reduction, no barrier);
//   * a rotary embedding of the trailing rope_dim channels, interleaved pairs
//     (2i, 2i+1), at position p = j*stride + offset.  The angle is reduced
//     exactly in turns: the frequency of pair i, theta^(-2i/rope_dim) / (2 pi)
//     turns per position, is a 64-bit fixed-point fraction of a turn that the
//     launcher evaluates once in double precision (a constant of theta and
//     rope_dim, passed by value: the GPU's FP64 units are far too slow to
//     evaluate it per thread); p times it modulo 2^64 -- an integer product --
//     is the angle's fraction of a turn, so the sine and cosine only ever see
//     an angle in [-pi, pi) (MUFU sin/cos, absolute error about 2^-21 there).
// The ratio-4 overlapping span (8 positions) is compiled with its span fixed;
// other spans take the general loop.
#include <math.h>

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

// Warp 0 finds the run of blockIdx.x: blockIdx.x counts chunks of E entries
// over the sequences in order, 32 sequences at a time (one load round trip
// each).  Writes the owning sequence (-1: past the last run) and the run's
// entry range [j0, j1).
__device__ __forceinline__ void locate_run(const int32_t* __restrict__ cu, int B, int r, int E, int* status,
                                           int* s_b, int* s_j0, int* s_j1) {
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
    *s_b = b;
    *s_j0 = c * E;
    *s_j1 = b >= 0 ? min(c * E + E, n) : 0;
  }
}

}  // namespace

constexpr int kMaxRopePairs = 256;

struct CompressExArgs {
  const void* x;
  const void* z;
  const void* xp;          // nullptr: one stream
  const void* zp;
  const float* P;
  const float* gamma;      // nullptr: no RMSNorm
  float eps;
  int rope_dim;            // 0: no rotary embedding
  int pos_stride, pos_offset;
  uint64_t rope_turn[kMaxRopePairs];  // pair i: theta^(-2i/rope_dim) / (2 pi) in units of 2^-64 turn
  const int32_t* cu;
  const int32_t* cu_cmp;
  int B, r, S, E, rows_max;
  void* out;
  int* status;
};

// kR, kS: the ratio and span when fixed at compile time (0: taken from a).
template <typename TIn, typename TOut, int D, int kR, int kS>
__global__ void __launch_bounds__(256) compress_ex_kernel(const __grid_constant__ CompressExArgs a) {
  constexpr int kPairs = D / 2;
  constexpr int kLanes = kPairs < 32 ? kPairs : 32;  // lanes per entry
  constexpr int kPerWarp = 32 / kLanes;              // entries per warp
  constexpr int kQ = kPairs / kLanes;                // channel pairs per lane
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_b, s_j0, s_j1;

  const int r = kR ? kR : a.r, S = kS ? kS : a.S;
  if (threadIdx.x < 32) locate_run(a.cu, a.B, r, a.E, a.status, &s_b, &s_j0, &s_j1);
  __syncthreads();
  const int b = s_b;
  if (b < 0) return;
  const int j0 = s_j0, j1 = s_j1;
  const bool two = a.xp != nullptr;
  const int tok0 = max(0, r * j0 + r - S);   // first local token the run reads
  const int tok1 = r * j1;                   // one past the last
  const int cur0 = two ? r * j0 : tok0;      // first token of the current-half rows
  const int Rc = tok1 - cur0;                // rows of x / z
  const int Rp = two ? tok1 - r - tok0 : 0;  // rows of x_prev / z_prev
  const int64_t seq0 = (int64_t)__ldg(a.cu + b);
  const int region = a.rows_max * D;
  TIn* sx = reinterpret_cast<TIn*>(smem);
  TIn* sz = sx + region;
  TIn* sxp = sz + region;
  TIn* szp = sxp + region;
  const uint32_t bar_a = smem_u32(&bar);

  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t bc = (uint32_t)Rc * D * sizeof(TIn), bp = (uint32_t)Rp * D * sizeof(TIn);
    mbar_arrive_expect_tx(bar_a, 2u * (bc + bp));
    constexpr uint32_t kPiece = 32768;
    const TIn* src[4] = {static_cast<const TIn*>(a.x) + (seq0 + cur0) * D,
                         static_cast<const TIn*>(a.z) + (seq0 + cur0) * D,
                         two ? static_cast<const TIn*>(a.xp) + (seq0 + tok0) * D : nullptr,
                         two ? static_cast<const TIn*>(a.zp) + (seq0 + tok0) * D : nullptr};
    TIn* dst[4] = {sx, sz, sxp, szp};
    for (int k = 0; k < 4; ++k) {
      const uint32_t bytes = k < 2 ? bc : bp;
      const char* g = reinterpret_cast<const char*>(src[k]);
      for (uint32_t off = 0; off < bytes; off += kPiece)
        bulk_g2s(smem_u32(dst[k]) + off, g + off, min(kPiece, bytes - off), bar_a);
    }
  }
  const bool ok = mbar_wait_bounded(bar_a, 0, a.status);
  if (__syncthreads_or(!ok)) return;

  const int lane = (int)threadIdx.x & 31, warp = (int)threadIdx.x >> 5;
  const int le = lane % kLanes, sub = lane / kLanes;
  const bool norm = a.gamma != nullptr;
  const int rope_lo = D - a.rope_dim;              // first rotated channel (D: none)
  const int usplit = two ? r : 0;                  // positions u < usplit read the previous half
  TOut* out = static_cast<TOut*>(a.out) + (int64_t)__ldg(a.cu_cmp + b) * D;
  const int n = j1 - j0;
  constexpr int kWarps = 256 / 32;
  for (int e0 = warp * kPerWarp; e0 < n; e0 += kWarps * kPerWarp) {  // uniform within a warp
    const int e = e0 + sub;
    const bool active = e < n;
    const int j = j0 + e;
    const int first = r * j + r - S;                 // span position u reads local token first + u
    const int ustart = active ? max(0, -first) : S;  // positions before the sequence start are left out
    // the row of span position u is base + u*D
    const TIn* xcur = sx + (first - cur0) * D;
    const TIn* zcur = sz + (first - cur0) * D;
    const TIn* xprv = two ? sxp + (first - tok0) * D : xcur;
    const TIn* zprv = two ? szp + (first - tok0) * D : zcur;
    float y[2 * kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int c = 2 * (le + q * kLanes);
      const float2* pcol = reinterpret_cast<const float2*>(a.P + c);
      float m0 = -INFINITY, m1 = -INFINITY, den0 = 0.f, den1 = 0.f, num0 = 0.f, num1 = 0.f;
      // a fixed span runs one masked pass from u = 0; otherwise chunks from ustart
      const int ubeg = kS ? 0 : ustart;
      for (int u0 = ubeg; u0 < S; u0 += 8) {
        float lg0[8], lg1[8], xv0[8], xv1[8];
        float cm0 = m0, cm1 = m1;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int u = u0 + k;
          lg0[k] = -INFINITY;
          lg1[k] = -INFINITY;
          xv0[k] = 0.f;
          xv1[k] = 0.f;
          if ((kS ? k < kS : u < S) && u >= ustart) {
            const bool pv = u < usplit;
            const float2 zz = load_pair((pv ? zprv : zcur) + u * D + c);
            const float2 xx = load_pair((pv ? xprv : xcur) + u * D + c);
            const float2 pp = __ldg(pcol + u * (D / 2));
            lg0[k] = zz.x + pp.x;
            lg1[k] = zz.y + pp.y;
            xv0[k] = xx.x;
            xv1[k] = xx.y;
            cm0 = fmaxf(cm0, lg0[k]);
            cm1 = fmaxf(cm1, lg1[k]);
          }
        }
        const float ms0 = -cm0 * kLog2e, ms1 = -cm1 * kLog2e;
        if (u0 != ubeg) {                            // rescale the running sums to the new maximum
          const float sc0 = ex2f(fmaf(m0, kLog2e, ms0)), sc1 = ex2f(fmaf(m1, kLog2e, ms1));
          den0 *= sc0;
          num0 *= sc0;
          den1 *= sc1;
          num1 *= sc1;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (kS && k >= kS) break;
          const float w0 = ex2f(fmaf(lg0[k], kLog2e, ms0)), w1 = ex2f(fmaf(lg1[k], kLog2e, ms1));
          den0 += w0;                                // a left-out position has weight 0
          den1 += w1;
          num0 = fmaf(w0, xv0[k], num0);
          num1 = fmaf(w1, xv1[k], num1);
        }
        m0 = cm0;
        m1 = cm1;
      }
      // den >= 1 (the maximum's own weight): the fast reciprocal divide is exact to 2 ulp
      y[2 * q] = active ? __fdividef(num0, den0) : 0.f;
      y[2 * q + 1] = active ? __fdividef(num1, den1) : 0.f;
    }
    if (norm) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 2 * kQ; ++k) ss = fmaf(y[k], y[k], ss);
#pragma unroll
      for (int o = kLanes / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = rsqrtf(ss * (1.0f / D) + a.eps);
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const float2 g = __ldg(reinterpret_cast<const float2*>(a.gamma + 2 * (le + q * kLanes)));
        y[2 * q] *= inv * g.x;
        y[2 * q + 1] *= inv * g.y;
      }
    }
    if (!active) continue;
    const int64_t p = (int64_t)j * a.pos_stride + a.pos_offset;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int c = 2 * (le + q * kLanes);
      float y0 = y[2 * q], y1 = y[2 * q + 1];
      if (c >= rope_lo) {
        // fraction of a turn (top 32 bits, signed: [-1/2, 1/2) turn) -> radians in [-pi, pi)
        const uint64_t ph = (uint64_t)p * a.rope_turn[(c - rope_lo) >> 1];
        const float ang = (float)(int32_t)(uint32_t)(ph >> 32) * 1.4629180792671596e-09f;  // 2 pi / 2^32
        float sn, cs;
        __sincosf(ang, &sn, &cs);
        const float t0 = y0 * cs - y1 * sn;
        y1 = y0 * sn + y1 * cs;
        y0 = t0;
      }
      store_pair(out + (int64_t)j * D + c, y0, y1);
    }
  }
}

// Staging rows and entries per CTA: about 64 span rows per run, fewer when
// `streams` staging buffers of that size would hold more than 40 KB (five
// CTAs per SM keep copies in flight while others reduce), but at least one
// entry per warp where the span allows.
static void compress_plan(int D, int r, int S, int in_bytes, int streams, int* rows_max, int* E, size_t* smem) {
  const size_t row_bytes = (size_t)streams * D * in_bytes;
  int e = S > 64 ? 1 : 64 / r;
  const long long fit = ((long long)(40 * 1024 / row_bytes) - (S - r)) / r;
  if (e > fit) e = (int)(fit < 1 ? 1 : fit);
  const int floor_e = S > 64 ? 1 : (64 / r < 8 ? 64 / r : 8);
  if (e < floor_e && row_bytes * (size_t)((S - r) + r * floor_e) <= 200 * 1024) e = floor_e;
  *E = e;
  *rows_max = (S - r) + r * e;
  *smem = row_bytes * (size_t)*rows_max;
}

bool compress_supported(int D, int r, int S, int in_bytes, bool two) {
  int rows, E;
  size_t smem;
  compress_plan(D, r, S, in_bytes, two ? 4 : 2, &rows, &E, &smem);
  return smem <= 200 * 1024 && (D == 32 || D == 64 || D == 128 || D == 256 || D == 512);
}

template <typename TIn, typename TOut, int D, int kR, int kS>
static cudaError_t launch_d(CompressExArgs& a, int T_cap, cudaStream_t stream) {
  size_t smem;
  compress_plan(D, a.r, a.S, (int)sizeof(TIn), a.xp ? 4 : 2, &a.rows_max, &a.E, &smem);
  auto kern = compress_ex_kernel<TIn, TOut, D, kR, kS>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long chunks = (long long)T_cap / ((long long)a.r * a.E) + a.B + 1;
  kern<<<(unsigned)chunks, 256, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int D>
static cudaError_t launch_span(CompressExArgs& a, int T_cap, cudaStream_t stream) {
  if (a.r == 4 && a.S == 8) return launch_d<TIn, TOut, D, 4, 8>(a, T_cap, stream);
  return launch_d<TIn, TOut, D, 0, 0>(a, T_cap, stream);
}

template <typename TIn, typename TOut>
static cudaError_t launch_t(CompressExArgs& a, int D, int T_cap, cudaStream_t stream) {
  switch (D) {
    case 32: return launch_span<TIn, TOut, 32>(a, T_cap, stream);
    case 64: return launch_span<TIn, TOut, 64>(a, T_cap, stream);
    case 128: return launch_span<TIn, TOut, 128>(a, T_cap, stream);
    case 256: return launch_span<TIn, TOut, 256>(a, T_cap, stream);
    case 512: return launch_span<TIn, TOut, 512>(a, T_cap, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_compress(const void* x, const void* z, const void* x_prev, const void* z_prev, const float* P,
                            const float* gamma, float eps, int rope_dim, float theta, int pos_stride,
                            int pos_offset, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap, int D,
                            int r, int S, bool fp32, void* out, int* status, cudaStream_t stream) {
  if (rope_dim / 2 > kMaxRopePairs) return cudaErrorInvalidValue;
  CompressExArgs a{x, z, x_prev, z_prev, P, gamma, eps, rope_dim, pos_stride, pos_offset, {},
                   cu, cu_cmp, B, r, S, 0, 0, out, status};
  for (int i = 0; i < rope_dim / 2; ++i) {
    // 2^64 / (2 pi) fixed-point turns per radian; the product stays below 2^63
    const double turns = pow((double)theta, -2.0 * i / rope_dim) * 2935890503282001226.0;
    a.rope_turn[i] = (uint64_t)llrint(turns);
  }
  if (fp32) return launch_t<float, float>(a, D, T_cap, stream);
  return launch_t<__nv_bfloat16, __nv_bfloat16>(a, D, T_cap, stream);
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
