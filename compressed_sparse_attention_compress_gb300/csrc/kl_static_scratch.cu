// kl_static_scratch.cu -- csa_indexer_kl for callers that cannot allocate.
//
// csa_indexer_kl needs a few bytes of device scratch per packed row (the
// per-query KL values and candidate counts that its fixed-order reduction
// reads back).  Some callers cannot hand it a workspace: code that runs where
// cudaMalloc is off limits (inside a CUDA-graph-captured region driven by a
// framework that owns every allocation, a real-time or memory-audited
// process, a plugin whose host forbids device allocations).  This entry point
// uses a scratch array that lives in the library's own device image instead.
//
// The array is a file-scope __device__ variable of fixed size, so every GPU
// that loads this library holds it (2 MiB) until the process exits.  Its
// device address is looked up once per device, with that device current,
// the first time the entry point runs on it; make that first call before any
// stream capture.  The address is cached for the life of the process, so it is
// stale after cudaDeviceReset or any other teardown of that device's primary
// context: do not call this entry point on the device again after one.  Calls
// share the array: two calls that overlap on the GPU
// (different streams, or different host threads) race on it and must be
// serialised by the caller.  Every scratch element a call reads is written
// earlier in the same call, so nothing in it has to start at zero and the
// contents a previous call left behind are never used.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/csa.h"

namespace csa {
int handle_device(csa_handle_t h);
}

namespace {

constexpr int kStaticMaxRows = 262144;                              // T_cap limit
constexpr size_t kStaticScratchBytes = (size_t)kStaticMaxRows * 8;  // float + int32 per row

static __device__ __align__(256) unsigned char g_kl_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_lock;
void* g_scratch_addr[kMaxDevices];  // device address of g_kl_scratch, per device

// Address of the scratch array on `device`; the device must be current.
csa_status_t scratch_on(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_addr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_kl_scratch);
    if (e != cudaSuccess || p == nullptr) return CSA_ERR_CUDA;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return CSA_OK;
}

}  // namespace

extern "C" csa_status_t csa_indexer_kl_static_scratch(
    csa_handle_t h, const void* q, const void* kv_cmp, const void* qI, const void* w, const void* kI,
    const int32_t* idx, int k_pad, const float* lse_cmp, const int32_t* cu, const int32_t* cu_cmp, int B,
    int T_cap, int max_seqlen, int H, int d, int H_I, int d_I, int ratio, float scale, csa_dtype_t dtype,
    float* kl_sum, float* kl_per_query, int32_t* n_valid, cudaStream_t stream) {
  if (h == nullptr || T_cap < 0) return CSA_ERR_INVALID_ARG;
  if (csa_indexer_kl_workspace(T_cap) > kStaticScratchBytes) return CSA_ERR_WORKSPACE;  // T_cap > 262144
  const int device = csa::handle_device(h);
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return CSA_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return CSA_ERR_CUDA;
  void* scratch = nullptr;
  const csa_status_t st = scratch_on(device, &scratch);
  if (prev != device) cudaSetDevice(prev);
  if (st != CSA_OK) return st;
  return csa_indexer_kl(h, q, kv_cmp, qI, w, kI, idx, k_pad, lse_cmp, cu, cu_cmp, B, T_cap, max_seqlen, H, d, H_I,
                        d_I, ratio, scale, dtype, kl_sum, kl_per_query, n_valid, scratch, kStaticScratchBytes,
                        stream);
}
