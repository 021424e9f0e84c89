// kl_blocks.cuh -- query blocks of the dense-teacher indexer KL kernels.
//
// "DeepSeek-V4 Attention Training Systems" §3: in the dense-loss phase C_t is
// every visible compressed entry of query t, a prefix of its sequence's
// compressed rows (entry j is visible once its block of r tokens has ended,
// j < (t + 1) / r).  Consecutive queries of one sequence share that prefix, so
// the forward and backward KL kernels both take blocks of QB consecutive
// queries and stream the block's longest prefix in tiles of TK entries.
#pragma once

#include <cstdint>

namespace csa {
namespace klb {

struct Block {
  int b;         // sequence
  int q0, nq;    // first query (within the sequence) and number of queries
  int seq0;      // packed row of the sequence's first query
  int cmp0;      // packed compressed row of the sequence's first entry
  int p0;        // position of the sequence's first row (context-parallel offset)
  int nvis_max;  // visible entries of the block's last query
  int ntiles;    // tiles of TK entries covering them
};

// Block k of all sequences' blocks, counted from the end of the packing, so
// that a persistent grid hands out the heaviest blocks (longest prefixes) first.
template <int QB, int TK>
__device__ __forceinline__ bool block_of(const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_cmp, int B,
                                         int r, int total, int k, Block& out, const int32_t* __restrict__ pos0) {
  int c = total - 1 - k;
  for (int bb = 0; bb < B; ++bb) {
    const int L = max(0, __ldg(cu + bb + 1) - __ldg(cu + bb));
    const int nb = (L + QB - 1) / QB;
    if (c < nb) {
      out.b = bb;
      out.q0 = c * QB;
      out.nq = min(QB, L - c * QB);
      out.seq0 = __ldg(cu + bb);
      out.cmp0 = __ldg(cu_cmp + bb);
      out.p0 = pos0 ? __ldg(pos0 + bb) : 0;
      out.nvis_max = (out.q0 + out.nq + out.p0) / r;
      out.ntiles = (out.nvis_max + TK - 1) / TK;
      return true;
    }
    c -= nb;
  }
  return false;
}

template <int QB>
__device__ __forceinline__ int total_blocks(const int32_t* __restrict__ cu, int B) {
  int n = 0;
  for (int bb = 0; bb < B; ++bb) n += (max(0, __ldg(cu + bb + 1) - __ldg(cu + bb)) + QB - 1) / QB;
  return n;
}

}  // namespace klb
}  // namespace csa
