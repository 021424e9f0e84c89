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
// One kernel serves csa_compress, csa_compress_ex and csa_compress_pair (both
// compressors of a layer in one launch).  The work is a list of runs -- E
// consecutive entries of one sequence -- whose raw rows are one contiguous span
// of each packed input stream.  A persistent CTA takes every gridDim-th run:
// its producer warp locates the run, and one lane stages the rows into a slot
// of a ring of shared-memory buffers with bulk asynchronous copies
// (cp.async.bulk, completion on the slot's mbarrier), keeping up to four runs
// in flight; eight consumer warps reduce the runs in order and release each
// slot on a second mbarrier.  Every input byte is read from HBM once per CTA
// and the overlap between neighbouring entries is served from shared memory.
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
// other spans take the general loop.  With that span, bf16 rows and none of
// the extras, a lane takes four adjacent channels (one 8-byte shared-memory
// read per row and stream) and does the softmax arithmetic on packed fp32
// pairs (add/fma .f32x2: two lanes of one instruction, each rounded exactly as
// the scalar operation), so the ALU work per element is about a third of the
// general loop's.  A span of 64 or more positions in runs of one entry (the
// ratio-128 compressor) is split across the consumer warps, which merge their
// partial softmax sums (maximum, sum of weights, weighted sum) through shared
// memory.
#include <math.h>
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace csa {

namespace {

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pairs: each half is rounded exactly as the scalar add / fma.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
      " add.rn.f32x2 pd, pa, pb;\n mov.b64 {%0, %1}, pd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 pa, pb, pc, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
      " mov.b64 pc, {%6, %7};\n fma.rn.f32x2 pd, pa, pb, pc;\n mov.b64 {%0, %1}, pd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) { return make_float2(bf16_lo(v), bf16_hi(v)); }

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

constexpr int kCuCache = 256;  // sequences whose offsets a CTA keeps in shared memory
constexpr int kConsumerWarps = 8;                    // warps that reduce entries
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kThreads = kConsumerThreads + 32;       // + the producer warp
constexpr int kMaxSlots = 4;                          // staging ring slots per CTA

// Warp 0: the run with index c (runs of E entries over the sequences in order,
// 32 sequences per load round trip) as (owning sequence or -1 past the last
// run, first entry j0, end entry j1, the sequence's first compressed row).
__device__ __forceinline__ int4 locate_run(const int32_t* cu, int B, int r, int E, int c, int* status) {
  const int lane = (int)threadIdx.x & 31;
  int b = -1, n = 0, ecarry = 0, cmp0 = 0;
  for (int base = 0; base < B && b < 0; base += 32) {
    const int bb = base + lane;
    int L = bb < B ? cu[bb + 1] - cu[bb] : 0;
    if (L < 0) { raise_status(status, CSA_ERR_DEVICE_BOUNDS); L = 0; }
    const int nb = L / r;
    const int nch = (nb + E - 1) / E;
    int incl = nch, ie = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      const int ve = __shfl_up_sync(0xffffffffu, ie, o);
      if (lane >= o) { incl += v; ie += ve; }
    }
    const uint32_t hit = __ballot_sync(0xffffffffu, bb < B && c < incl);
    if (hit != 0u) {
      const int w = __ffs(hit) - 1;  // first sequence whose runs reach c
      b = base + w;
      c -= __shfl_sync(0xffffffffu, incl - nch, w);
      n = __shfl_sync(0xffffffffu, nb, w);
      cmp0 = ecarry + __shfl_sync(0xffffffffu, ie - nb, w);
    } else {
      c -= __shfl_sync(0xffffffffu, incl, 31);
      ecarry += __shfl_sync(0xffffffffu, ie, 31);
    }
  }
  return make_int4(b, c * E, b >= 0 ? min(c * E + E, n) : 0, cmp0);
}

// Warp 0: the number of runs of E entries over all sequences.
__device__ __forceinline__ int count_runs(const int32_t* cu, int B, int r, int E) {
  const int lane = (int)threadIdx.x & 31;
  int total = 0;
  for (int base = 0; base < B; base += 32) {
    const int bb = base + lane;
    const int L = bb < B ? max(0, cu[bb + 1] - cu[bb]) : 0;
    total += (L / r + E - 1) / E;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  return total;
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
  const int32_t* cu;
  const int32_t* cu_cmp;
  int B, r, S, E, rows_max;
  void* out;
  int* status;
};

// The rotary frequencies of stream 0, a separate kernel parameter after both
// streams' scalars and pointers: pair i turns theta^(-2i/rope_dim) / (2 pi) of a turn per position, in units
// of 2^-64 turn.
struct RopeTurns {
  uint64_t t[kMaxRopePairs];
};

// The raw rows run `ri` reads, one contiguous span of each packed input stream:
// x and z from the current-half rows on, x_prev and z_prev (when given) from
// the run's first token on.  Staging layout: [x | z | x_prev | z_prev], each
// rows_max x D.
struct RunRows {
  int tok0, cur0, Rc, Rp;
};
__device__ __forceinline__ RunRows run_rows(const CompressExArgs& a, int r, int S, int4 ri) {
  const bool two = a.xp != nullptr;
  const int tok0 = max(0, r * ri.y + r - S);  // first local token the run reads
  const int tok1 = r * ri.z;                  // one past the last
  const int cur0 = two ? r * ri.y : tok0;     // first token of the current-half rows
  return RunRows{tok0, cur0, tok1 - cur0, two ? tok1 - r - tok0 : 0};
}

// Thread 0: bulk copies of the run's rows into `buf`, completing on `bar`.
template <typename TIn, int D>
__device__ __forceinline__ void stage_run(const CompressExArgs& a, int r, int S, int4 ri, int64_t seq0, uint32_t buf,
                                          uint32_t bar) {
  const RunRows rr = run_rows(a, r, S, ri);
  const bool two = a.xp != nullptr;
  const uint32_t region = (uint32_t)a.rows_max * D * sizeof(TIn);
  const uint32_t bc = (uint32_t)rr.Rc * D * sizeof(TIn), bp = (uint32_t)rr.Rp * D * sizeof(TIn);
  mbar_arrive_expect_tx(bar, 2u * (bc + bp));
  constexpr uint32_t kPiece = 32768;
  const TIn* src[4] = {static_cast<const TIn*>(a.x) + (seq0 + rr.cur0) * D,
                       static_cast<const TIn*>(a.z) + (seq0 + rr.cur0) * D,
                       two ? static_cast<const TIn*>(a.xp) + (seq0 + rr.tok0) * D : nullptr,
                       two ? static_cast<const TIn*>(a.zp) + (seq0 + rr.tok0) * D : nullptr};
  for (int k = 0; k < 4; ++k) {
    const uint32_t bytes = k < 2 ? bc : bp;
    const char* g = reinterpret_cast<const char*>(src[k]);
    for (uint32_t off = 0; off < bytes; off += kPiece)
      bulk_g2s(buf + k * region + off, g + off, min(kPiece, bytes - off), bar);
  }
}

// One entry's four channels [c, c+4) over a fixed span of kS positions: zrow
// / xrow point at span position 0's staged rows (row stride D), pcol at P's
// column c.  kMask: positions u < ustart lie before the sequence start; their
// rows are not staged and they are left out (weight 0).
template <int D, int kS, bool kMask, typename TOut>
__device__ __forceinline__ void plain_entry4(const __nv_bfloat16* zrow, const __nv_bfloat16* xrow,
                                             const float* pcol, int ustart, TOut* dst) {
  constexpr float kLog2e = 1.4426950408889634f;
  float2 la[kS], lb[kS];  // logits of channels (c, c+1) and (c+2, c+3)
  uint2 xv[kS];
#pragma unroll
  for (int u = 0; u < kS; ++u) {
    if (!kMask || u >= ustart) {
      const uint2 zz = *reinterpret_cast<const uint2*>(zrow + u * D);
      xv[u] = *reinterpret_cast<const uint2*>(xrow + u * D);
      const float4 pp = __ldg(reinterpret_cast<const float4*>(pcol + u * D));
      la[u] = add2(unpack_bf16x2(zz.x), make_float2(pp.x, pp.y));
      lb[u] = add2(unpack_bf16x2(zz.y), make_float2(pp.z, pp.w));
    } else {
      la[u] = lb[u] = make_float2(-INFINITY, -INFINITY);
      xv[u] = make_uint2(0u, 0u);
    }
  }
  float m[4] = {la[0].x, la[0].y, lb[0].x, lb[0].y};
#pragma unroll
  for (int u = 1; u < kS; u += 2) {
    if (u + 1 < kS) {
      m[0] = max3f(m[0], la[u].x, la[u + 1].x);
      m[1] = max3f(m[1], la[u].y, la[u + 1].y);
      m[2] = max3f(m[2], lb[u].x, lb[u + 1].x);
      m[3] = max3f(m[3], lb[u].y, lb[u + 1].y);
    } else {
      m[0] = fmaxf(m[0], la[u].x);
      m[1] = fmaxf(m[1], la[u].y);
      m[2] = fmaxf(m[2], lb[u].x);
      m[3] = fmaxf(m[3], lb[u].y);
    }
  }
  const float2 l2 = make_float2(kLog2e, kLog2e);
  const float2 msa = make_float2(-m[0] * kLog2e, -m[1] * kLog2e), msb = make_float2(-m[2] * kLog2e, -m[3] * kLog2e);
  float2 da = make_float2(0.f, 0.f), db = da, na = da, nb = da;
#pragma unroll
  for (int u = 0; u < kS; ++u) {
    const float2 ta = fma2(la[u], l2, msa), tb = fma2(lb[u], l2, msb);
    const float2 wa = make_float2(ex2f(ta.x), ex2f(ta.y)), wb = make_float2(ex2f(tb.x), ex2f(tb.y));
    da = add2(da, wa);                              // a left-out position has weight 0
    db = add2(db, wb);
    na = fma2(wa, unpack_bf16x2(xv[u].x), na);
    nb = fma2(wb, unpack_bf16x2(xv[u].y), nb);
  }
  // den >= 1 (the maximum's own weight): the fast reciprocal divide is exact to 2 ulp
  const float y0 = __fdividef(na.x, da.x), y1 = __fdividef(na.y, da.y);
  const float y2 = __fdividef(nb.x, db.x), y3 = __fdividef(nb.y, db.y);
  if constexpr (std::is_same<TOut, float>::value) {
    *reinterpret_cast<float4*>(dst) = make_float4(y0, y1, y2, y3);
  } else {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
  }
}

// All threads: the entries of run `ri` (one stream, fixed span kS, bf16 rows,
// no extras) from the rows staged at sx / sz, four channels per lane.
template <typename TOut, int D, int kS>
__device__ __forceinline__ void compress_run_plain(const CompressExArgs& a, int4 ri, int r, int cur0,
                                                   const __nv_bfloat16* sx, const __nv_bfloat16* sz) {
  constexpr int kLanes = D / 4 < 32 ? D / 4 : 32;  // lanes per entry
  constexpr int kPerWarp = 32 / kLanes;            // entries per warp
  constexpr int kQ = D / 4 / kLanes;               // four-channel groups per lane
  constexpr int kWarps = kConsumerWarps;
  const int lane = (int)threadIdx.x & 31, warp = (int)threadIdx.x >> 5;
  const int le = lane % kLanes, sub = lane / kLanes;
  const int n = ri.z - ri.y;
  TOut* out = static_cast<TOut*>(a.out) + (int64_t)ri.w * D;
  for (int e = warp * kPerWarp + sub; e < n; e += kWarps * kPerWarp) {  // no warp-collective work inside
    const int j = ri.y + e;
    const int first = r * j + r - kS;  // span position u reads local token first + u
    const int ustart = max(0, -first);
    const int row0 = first - cur0;     // its staged row (rows below 0 are never read)
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int c = 4 * (le + q * kLanes);
      const __nv_bfloat16* zrow = sz + row0 * D + c;
      const __nv_bfloat16* xrow = sx + row0 * D + c;
      if (ustart == 0)
        plain_entry4<D, kS, false>(zrow, xrow, a.P + c, 0, out + (int64_t)j * D + c);
      else
        plain_entry4<D, kS, true>(zrow, xrow, a.P + c, ustart, out + (int64_t)j * D + c);
    }
  }
}

// The consumer warps meet at `bar` (an mbarrier counting one arrival per
// consumer warp; `phase` counts the meetings this thread has passed).  Bounded:
// false, with the status word set, when a warp does not come.
__device__ __forceinline__ bool consumers_meet(uint32_t bar, uint32_t& phase, int* status) {
  __syncwarp();
  if (((int)threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, phase & 1u, status));
  ++phase;
  return ok;
}

// Consumer threads: the entries of run `ri` from its rows staged in
// `smem_buf`.  kR, kS: the ratio and span when fixed at compile time (0: taken
// from a).  sync_bar / sync_phase: the consumers' meeting barrier (the split
// path of a long span uses it twice per run).
template <typename TIn, typename TOut, int D, int kR, int kS>
__device__ __forceinline__ void compress_run(const CompressExArgs& a, const uint64_t* rope_turn, int4 ri,
                                             const uint8_t* smem_buf, uint32_t sync_bar, uint32_t& sync_phase) {
  constexpr int kPairs = D / 2;
  constexpr int kLanes = kPairs < 32 ? kPairs : 32;  // lanes per entry
  constexpr int kPerWarp = 32 / kLanes;              // entries per warp
  constexpr int kQ = kPairs / kLanes;                // channel pairs per lane
  constexpr float kLog2e = 1.4426950408889634f;
  const int r = kR ? kR : a.r, S = kS ? kS : a.S;
  const bool two = a.xp != nullptr;
  const RunRows rr = run_rows(a, r, S, ri);
  const int tok0 = rr.tok0, cur0 = rr.cur0;
  const int j0 = ri.y, j1 = ri.z;
  const int region = a.rows_max * D;
  const TIn* sx = reinterpret_cast<const TIn*>(smem_buf);
  const TIn* sz = sx + region;
  const TIn* sxp = sz + region;
  const TIn* szp = sxp + region;
  const int lane = (int)threadIdx.x & 31, warp = (int)threadIdx.x >> 5;
  const int le = lane % kLanes, sub = lane / kLanes;
  const bool norm = a.gamma != nullptr;
  const int rope_lo = D - a.rope_dim;              // first rotated channel (D: none)
  const int usplit = two ? r : 0;                  // positions u < usplit read the previous half
  TOut* out = static_cast<TOut*>(a.out) + (int64_t)ri.w * D;
  const int n = j1 - j0;
  constexpr int kWarps = kConsumerWarps;
  if constexpr (kS > 0 && kS <= 8 && std::is_same<TIn, __nv_bfloat16>::value && D >= 16) {
    if (!two && !norm && a.rope_dim == 0) {
      compress_run_plain<TOut, D, kS>(a, ri, r, cur0, sx, sz);
      return;
    }
  }
  if (S >= 64 && n == 1 && a.E == 1) {
    // one long span per run (ratio 128): warp w reduces the span positions
    // [w S/8, (w+1) S/8) of the entry, then warp 0 merges the eight partial
    // softmax sums (max, sum of weights, weighted sum) and finishes the entry
    const int j = j0;
    const int first = r * j + r - S;
    const int per = S / kWarps;
    const int ulo = max(warp * per, max(0, -first)), uhi = (warp + 1) * per;
    const TIn* xcur = sx + (first - cur0) * D;
    const TIn* zcur = sz + (first - cur0) * D;
    const TIn* xprv = two ? sxp + (first - tok0) * D : xcur;
    const TIn* zprv = two ? szp + (first - tok0) * D : zcur;
    float pm[2 * kQ], pd[2 * kQ], pn[2 * kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int c = 2 * (le + q * kLanes);
      const float2* pcol = reinterpret_cast<const float2*>(a.P + c);
      float m0 = -INFINITY, m1 = -INFINITY, d0 = 0.f, d1 = 0.f, n0 = 0.f, n1 = 0.f;
      for (int u = ulo; u < uhi; ++u) {
        const bool pv = u < usplit;
        const float2 zz = load_pair((pv ? zprv : zcur) + u * D + c);
        const float2 xx = load_pair((pv ? xprv : xcur) + u * D + c);
        const float2 pp = __ldg(pcol + u * (D / 2));
        const float l0 = zz.x + pp.x, l1 = zz.y + pp.y;
        if (l0 > m0) {  // a new maximum: rescale the sums (m0 = -inf: they are 0)
          const float sc = ex2f((m0 - l0) * kLog2e);
          d0 *= sc;
          n0 *= sc;
          m0 = l0;
        }
        if (l1 > m1) {
          const float sc = ex2f((m1 - l1) * kLog2e);
          d1 *= sc;
          n1 *= sc;
          m1 = l1;
        }
        const float w0 = ex2f((l0 - m0) * kLog2e), w1 = ex2f((l1 - m1) * kLog2e);
        d0 += w0;
        d1 += w1;
        n0 = fmaf(w0, xx.x, n0);
        n1 = fmaf(w1, xx.y, n1);
      }
      pm[2 * q] = m0; pm[2 * q + 1] = m1;
      pd[2 * q] = d0; pd[2 * q + 1] = d1;
      pn[2 * q] = n0; pn[2 * q + 1] = n1;
    }
    // every warp has read the staged rows: the partials go over them
    if (!consumers_meet(sync_bar, sync_phase, a.status)) return;
    float* part = reinterpret_cast<float*>(const_cast<uint8_t*>(smem_buf));  // [warp][channel][3]
    if (lane < kLanes) {
#pragma unroll
      for (int q = 0; q < kQ; ++q)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float* pp = part + ((size_t)warp * D + 2 * (le + q * kLanes) + h) * 3;
          pp[0] = pm[2 * q + h];
          pp[1] = pd[2 * q + h];
          pp[2] = pn[2 * q + h];
        }
    }
    fence_proxy_async_shared();  // these generic writes come before the slot's next bulk copies
    if (!consumers_meet(sync_bar, sync_phase, a.status)) return;
    if (warp != 0 || lane >= kLanes) return;
    float y[2 * kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = 2 * (le + q * kLanes) + h;
        float m = -INFINITY;
        for (int w = 0; w < kWarps; ++w) m = fmaxf(m, part[((size_t)w * D + c) * 3]);
        float den = 0.f, num = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          const float* pp = part + ((size_t)w * D + c) * 3;
          if (pp[0] == -INFINITY) continue;  // a warp whose positions were all left out
          const float sc = ex2f((pp[0] - m) * kLog2e);
          den = fmaf(pp[1], sc, den);
          num = fmaf(pp[2], sc, num);
        }
        y[2 * q + h] = __fdividef(num, den);  // den >= 1: the maximum's own weight
      }
    if (norm) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 2 * kQ; ++k) ss = fmaf(y[k], y[k], ss);
      const uint32_t mask = kLanes == 32 ? 0xffffffffu : ((1u << kLanes) - 1u);
#pragma unroll
      for (int o = kLanes / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(mask, ss, o);
      const float inv = rsqrtf(ss * (1.0f / D) + a.eps);
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const float2 g = __ldg(reinterpret_cast<const float2*>(a.gamma + 2 * (le + q * kLanes)));
        y[2 * q] *= inv * g.x;
        y[2 * q + 1] *= inv * g.y;
      }
    }
    const int64_t p = (int64_t)j * a.pos_stride + a.pos_offset;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int c = 2 * (le + q * kLanes);
      float y0 = y[2 * q], y1 = y[2 * q + 1];
      if (c >= rope_lo) {
        const uint64_t ph = (uint64_t)p * rope_turn[(c - rope_lo) >> 1];
        const float ang = (float)(int32_t)(uint32_t)(ph >> 32) * 1.4629180792671596e-09f;  // 2 pi / 2^32
        float sn, cs;
        __sincosf(ang, &sn, &cs);
        const float t0 = y0 * cs - y1 * sn;
        y1 = y0 * sn + y1 * cs;
        y0 = t0;
      }
      store_pair(out + (int64_t)j * D + c, y0, y1);
    }
    return;
  }
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
        const uint64_t ph = (uint64_t)p * rope_turn[(c - rope_lo) >> 1];
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

// One CTA processes runs g = blockIdx.x + i * gridDim.x of a combined list --
// the runs of stream a0, then (D1 > 0) those of stream a1.  The last warp is
// the producer: it locates each run, waits for a free slot of a ring of
// `nslot` staging buffers, writes the run's metadata beside it and starts the
// bulk copies of its rows, so up to nslot runs are in flight.  The consumer
// warps reduce the runs in order, each waiting for its slot's copies and
// releasing the slot when done -- no CTA-wide barrier between runs.  The
// producer ends the list with a sentinel run, writes the compressed offsets
// (block 0, when cu_cmp_out is given), and waits for every copy it started
// before it leaves.
template <typename TIn, typename TOut, int D0, int D1, int kR, int kS>
__global__ void __launch_bounds__(kThreads, (D0 <= 128 ? 3 : 1))
    compress_kernel(const __grid_constant__ CompressExArgs a0, const __grid_constant__ CompressExArgs a1,
                    uint32_t buf_bytes, int nslot, int32_t* __restrict__ cu_cmp_out,
                    const __grid_constant__ RopeTurns rope) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t s_full[kMaxSlots];
  __shared__ __align__(8) uint64_t s_empty[kMaxSlots];
  __shared__ __align__(8) uint64_t s_meet;
  __shared__ int4 s_run[kMaxSlots];
  __shared__ int s_which[kMaxSlots];
  __shared__ int32_t s_cu[kCuCache + 1];  // the packing's offsets (producer), on chip when B is small
  const int tid = (int)threadIdx.x;
  const int lane = tid & 31;
  const int r = kR ? kR : a0.r, S = kS ? kS : a0.S;
  if (tid == 0) {
    for (int k = 0; k < nslot; ++k) {
      mbar_init(smem_u32(&s_full[k]), 1);
      mbar_init(smem_u32(&s_empty[k]), kConsumerWarps);
    }
    mbar_init(smem_u32(&s_meet), kConsumerWarps);
    fence_mbar_init();
  }
  __syncthreads();  // the only barrier of the whole CTA
  if (tid >= kConsumerThreads) {
    // ---------------- producer warp ----------------
    const bool cached = a0.B <= kCuCache;
    if (cached) {
      for (int i = lane; i <= a0.B; i += 32) s_cu[i] = __ldg(a0.cu + i);
      __syncwarp();
    }
    const int32_t* cu = cached ? s_cu : a0.cu;  // both streams share the packing
    const int n0 = D1 > 0 ? count_runs(cu, a0.B, r, a0.E) : 0x7fffffff;
    int k = 0;         // runs pushed (the sentinel not counted)
    bool failed = false;
    for (;; ++k) {
      const int g = blockIdx.x + k * (int)gridDim.x;
      int4 ri;
      int which = 0;
      if (g < n0) {
        ri = locate_run(cu, a0.B, r, a0.E, g, a0.status);
      } else {
        ri = locate_run(cu, a1.B, r, a1.E, g - n0, a1.status);
        which = 1;
      }
      const int slot = k % nslot;
      const uint32_t use = (uint32_t)(k / nslot);
      // the slot's previous run (push k - nslot) has been released by every consumer warp
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&s_empty[slot]), (use & 1u) ^ 1u, a0.status))) {
        failed = true;
        break;
      }
      if (lane == 0) {
        s_run[slot] = ri;
        s_which[slot] = which;
        if (ri.x < 0) {
          mbar_arrive(smem_u32(&s_full[slot]));  // the sentinel: no copies
        } else {
          fence_proxy_async_shared();
          const uint32_t buf = smem_u32(smem) + (uint32_t)slot * buf_bytes, bar = smem_u32(&s_full[slot]);
          const int64_t seq0 = cu[ri.x];
          if (which == 0) stage_run<TIn, D0>(a0, r, S, ri, seq0, buf, bar);
          if constexpr (D1 > 0) {
            if (which == 1) stage_run<TIn, D1>(a1, r, S, ri, seq0, buf, bar);
          }
        }
      }
      __syncwarp();
      if (ri.x < 0) break;  // uniform: every lane located the same run
    }
    if (blockIdx.x == 0 && cu_cmp_out != nullptr) {  // cu_cmp[b] = sum_{b' < b} floor(L_b' / r)
      int carry = 0;
      if (lane == 0) {
        cu_cmp_out[0] = 0;
        if (cu[0] != 0) raise_status(a0.status, CSA_ERR_DEVICE_BOUNDS);
      }
      for (int base = 0; base < a0.B; base += 32) {
        const int bb = base + lane;
        const int n = bb < a0.B ? max(0, cu[bb + 1] - cu[bb]) / r : 0;
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (bb < a0.B) cu_cmp_out[bb + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    // leave no copy in flight into this CTA's shared memory: pushes k - nslot + 1 .. k - 1
    // (and k - nslot, whose release was not seen, after a failed wait)
    for (int q = max(0, k - nslot + (failed ? 0 : 1)); q < k; ++q)
      mbar_wait_bounded(smem_u32(&s_full[q % nslot]), (uint32_t)(q / nslot) & 1u, a0.status);
    return;
  }
  // ---------------- consumer warps ----------------
  uint32_t meet_phase = 0;
  for (int k = 0;; ++k) {
    const int slot = k % nslot;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&s_full[slot]), (uint32_t)(k / nslot) & 1u, a0.status)))
      return;
    const int4 ri = s_run[slot];
    const int which = s_which[slot];
    if (ri.x < 0) return;  // the sentinel
    const uint8_t* buf = smem + (size_t)slot * buf_bytes;
    if (which == 0) compress_run<TIn, TOut, D0, kR, kS>(a0, rope.t, ri, buf, smem_u32(&s_meet), meet_phase);
    if constexpr (D1 > 0) {
      if (which == 1) compress_run<TIn, TOut, D1, kR, kS>(a1, rope.t, ri, buf, smem_u32(&s_meet), meet_phase);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s_empty[slot]));
  }
}

// Staging rows and entries per run: about 64 span rows, fewer when `streams`
// staging buffers of that size would hold more than 32 KB (each CTA holds two
// runs' rows, and three CTAs per SM keep copies in flight while others
// reduce), but at least one entry per warp where the span allows.  per_round
// > 0 (the plain fixed-span path): exactly one pass of the CTA's warps, so no
// warp waits at the end of a run for another's second entry.
static void compress_plan(int D, int r, int S, int in_bytes, int streams, int per_round, int* rows_max, int* E,
                          size_t* smem) {
  const size_t row_bytes = (size_t)streams * D * in_bytes;
  int e = S > 64 ? 1 : 64 / r;
  const long long fit = ((long long)(32 * 1024 / row_bytes) - (S - r)) / r;
  if (e > fit) e = (int)(fit < 1 ? 1 : fit);
  const int floor_e = S > 64 ? 1 : (64 / r < 8 ? 64 / r : 8);
  if (e < floor_e && row_bytes * (size_t)((S - r) + r * floor_e) <= 200 * 1024) e = floor_e;
  if (per_round > 0 && row_bytes * (size_t)((S - r) + r * per_round) <= 100 * 1024) e = per_round;
  *E = e;
  *rows_max = (S - r) + r * e;
  *smem = row_bytes * (size_t)*rows_max;
}

// The plain fixed-span path of compress_run (ratio 4, span 8, bf16 rows, one
// stream, no RMSNorm or rotary embedding) and the entries one pass of a CTA's
// warps reduces there (an entry takes min(32, D/4) lanes); 0 otherwise.
static int plain_round(const CompressExArgs& a, int D, int in_bytes) {
  const bool plain = a.r == 4 && a.S == 8 && in_bytes == 2 && a.xp == nullptr && a.gamma == nullptr &&
                     a.rope_dim == 0 && D >= 16;
  return plain ? kConsumerWarps * (32 / (D / 4 < 32 ? D / 4 : 32)) : 0;
}

bool compress_supported(int D, int r, int S, int in_bytes, bool two) {
  int rows, E;
  size_t smem;
  compress_plan(D, r, S, in_bytes, two ? 4 : 2, 0, &rows, &E, &smem);
  return smem <= 200 * 1024 && (D == 32 || D == 64 || D == 128 || D == 256 || D == 512);
}

// Staging ring slots per CTA: as many as fit in 128 KB (at least one, at
// most kMaxSlots); the kernel's shared-memory attributes, and the grid of the
// persistent kernel: the CTAs that are resident at once (by registers, threads
// and shared memory), at most one per run.
static int compress_slots(size_t buf_bytes) {
  const size_t n = (size_t)(128 * 1024) / buf_bytes;
  return n < 1 ? 1 : (n > (size_t)kMaxSlots ? kMaxSlots : (int)n);
}
template <typename K>
static cudaError_t compress_setup(K kern, size_t dyn_smem, long long runs, unsigned* grid) {
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_smem);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0, per_sm = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, dyn_smem)) != cudaSuccess)
    return err;
  const long long slots = (long long)(per_sm < 1 ? 1 : per_sm) * sms;
  *grid = (unsigned)(runs < slots ? (runs > 0 ? runs : 1) : slots);
  return cudaSuccess;
}

template <typename TIn, typename TOut, int D, int kR, int kS>
static cudaError_t launch_d(CompressExArgs& a, const RopeTurns& rope, int T_cap, cudaStream_t stream) {
  size_t smem;
  compress_plan(D, a.r, a.S, (int)sizeof(TIn), a.xp ? 4 : 2, plain_round(a, D, (int)sizeof(TIn)), &a.rows_max, &a.E,
                &smem);
  auto kern = compress_kernel<TIn, TOut, D, 0, kR, kS>;
  const int nslot = compress_slots(smem);
  const long long runs = (long long)T_cap / ((long long)a.r * a.E) + a.B + 1;  // an upper bound
  unsigned grid = 1;
  const cudaError_t err = compress_setup(kern, nslot * smem, runs, &grid);
  if (err != cudaSuccess) return err;
  kern<<<grid, kThreads, nslot * smem, stream>>>(a, a, (uint32_t)smem, nslot, nullptr, rope);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int D>
static cudaError_t launch_span(CompressExArgs& a, const RopeTurns& rope, int T_cap, cudaStream_t stream) {
  if (a.r == 4 && a.S == 8) return launch_d<TIn, TOut, D, 4, 8>(a, rope, T_cap, stream);
  return launch_d<TIn, TOut, D, 0, 0>(a, rope, T_cap, stream);
}

template <typename TIn, typename TOut>
static cudaError_t launch_t(CompressExArgs& a, const RopeTurns& rope, int D, int T_cap, cudaStream_t stream) {
  switch (D) {
    case 32: return launch_span<TIn, TOut, 32>(a, rope, T_cap, stream);
    case 64: return launch_span<TIn, TOut, 64>(a, rope, T_cap, stream);
    case 128: return launch_span<TIn, TOut, 128>(a, rope, T_cap, stream);
    case 256: return launch_span<TIn, TOut, 256>(a, rope, T_cap, stream);
    case 512: return launch_span<TIn, TOut, 512>(a, rope, T_cap, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_compress(const void* x, const void* z, const void* x_prev, const void* z_prev, const float* P,
                            const float* gamma, float eps, int rope_dim, float theta, int pos_stride,
                            int pos_offset, const int32_t* cu, const int32_t* cu_cmp, int B, int T_cap, int D,
                            int r, int S, bool fp32, void* out, int* status, cudaStream_t stream) {
  if (rope_dim / 2 > kMaxRopePairs) return cudaErrorInvalidValue;
  CompressExArgs a{x, z, x_prev, z_prev, P, gamma, eps, rope_dim, pos_stride, pos_offset,
                   cu, cu_cmp, B, r, S, 0, 0, out, status};
  RopeTurns rope{};
  for (int i = 0; i < rope_dim / 2; ++i) {
    // 2^64 / (2 pi) fixed-point turns per radian; the product stays below 2^63
    const double turns = pow((double)theta, -2.0 * i / rope_dim) * 2935890503282001226.0;
    rope.t[i] = (uint64_t)llrint(turns);
  }
  if (fp32) return launch_t<float, float>(a, rope, D, T_cap, stream);
  return launch_t<__nv_bfloat16, __nv_bfloat16>(a, rope, D, T_cap, stream);
}

template <typename TIn, typename TOut, int D0, int D1, int kR, int kS>
static cudaError_t launch_pair_d(CompressExArgs& a0, CompressExArgs& a1, int T_cap, int32_t* cu_cmp,
                                 cudaStream_t stream) {
  size_t s0, s1;
  const int in_bytes = (int)sizeof(TIn);
  compress_plan(D0, a0.r, a0.S, in_bytes, 2, plain_round(a0, D0, in_bytes), &a0.rows_max, &a0.E, &s0);
  compress_plan(D1, a1.r, a1.S, in_bytes, 2, plain_round(a1, D1, in_bytes), &a1.rows_max, &a1.E, &s1);
  const size_t smem = s0 > s1 ? s0 : s1;
  auto kern = compress_kernel<TIn, TOut, D0, D1, kR, kS>;
  const int nslot = compress_slots(smem);
  const long long runs = (long long)T_cap / ((long long)a0.r * a0.E) + (long long)T_cap / ((long long)a1.r * a1.E) +
                         2 * (long long)a0.B + 2;  // an upper bound
  unsigned grid = 1;
  const cudaError_t err = compress_setup(kern, nslot * smem, runs, &grid);
  if (err != cudaSuccess) return err;
  kern<<<grid, kThreads, nslot * smem, stream>>>(a0, a1, (uint32_t)smem, nslot, cu_cmp, RopeTurns{});
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int D0, int D1>
static cudaError_t launch_pair_span(CompressExArgs& a0, CompressExArgs& a1, int T_cap, int32_t* cu_cmp,
                                    cudaStream_t stream) {
  if (a0.r == 4 && a0.S == 8) return launch_pair_d<TIn, TOut, D0, D1, 4, 8>(a0, a1, T_cap, cu_cmp, stream);
  return launch_pair_d<TIn, TOut, D0, D1, 0, 0>(a0, a1, T_cap, cu_cmp, stream);
}

bool compress_pair_supported(int D, int D_I, int r, int S, int in_bytes) {
  return ((D == 128 && D_I == 64) || (D == 64 && D_I == 32)) && compress_supported(D, r, S, in_bytes, false) &&
         compress_supported(D_I, r, S, in_bytes, false);
}

cudaError_t launch_compress_pair(const void* x, const void* z, const float* P, void* out, int D, const void* x_i,
                                 const void* z_i, const float* P_i, void* out_i, int D_I, const int32_t* cu, int B,
                                 int T_cap, int r, int S, bool fp32, int32_t* cu_cmp, int* status,
                                 cudaStream_t stream) {
  CompressExArgs a0{x, z, nullptr, nullptr, P, nullptr, 0.f, 0, 0, 0, cu, cu_cmp, B, r, S, 0, 0, out, status};
  CompressExArgs a1{x_i, z_i, nullptr, nullptr, P_i, nullptr, 0.f, 0, 0, 0, cu, cu_cmp, B, r, S, 0, 0, out_i,
                    status};
  if (D == 128 && D_I == 64)
    return fp32 ? launch_pair_span<float, float, 128, 64>(a0, a1, T_cap, cu_cmp, stream)
                : launch_pair_span<__nv_bfloat16, __nv_bfloat16, 128, 64>(a0, a1, T_cap, cu_cmp, stream);
  if (D == 64 && D_I == 32)
    return fp32 ? launch_pair_span<float, float, 64, 32>(a0, a1, T_cap, cu_cmp, stream)
                : launch_pair_span<__nv_bfloat16, __nv_bfloat16, 64, 32>(a0, a1, T_cap, cu_cmp, stream);
  return cudaErrorInvalidValue;
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
