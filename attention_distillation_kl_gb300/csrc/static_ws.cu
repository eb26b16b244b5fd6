// Key-split forward for callers that cannot allocate device memory.
//
// streamkl_fwd_splitk needs a caller-owned workspace for the per-split
// partial statistics.  Some callers have no way to provide one: code running
// under a framework whose caching allocator owns all device memory (calling
// cudaMalloc behind its back can synchronise the device and break its
// accounting), or host runtimes that must not fail for lack of memory in the
// middle of a step.  For them this file keeps the partials in one fixed
// device array that belongs to the library, and the entry point allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// The array is a file-scope __device__ object of STREAMKL_STATIC_WORKSPACE_BYTES,
// so every GPU on which the library's module is loaded holds that much memory
// until the process exits.  In host code its name is only a host-side stand-in
// for the symbol, never a device address: the device address is looked up
// with cudaGetSymbolAddress on every call, on the current device.
#include <cuda_runtime.h>

#include "streamkl.h"

namespace {

constexpr size_t kStaticFloats = STREAMKL_STATIC_WORKSPACE_BYTES / sizeof(float);

// Shared by every call on a device; the contents of the last call remain.
static __device__ __align__(256) float g_splitk_static_ws[kStaticFloats];

// Device address of g_splitk_static_ws on the current device, looked up on
// every call (cheap, and never stale: a cudaDeviceReset reloads the module
// and may move the array).  Returns STREAMKL_OK and sets *out.
int static_ws_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_splitk_static_ws);
  if (e != cudaSuccess || p == nullptr) return STREAMKL_CUDA_ERROR;
  *out = p;
  return STREAMKL_OK;
}

}  // namespace

extern "C" int streamkl_fwd_splitk_noalloc(const void* q1, const void* k1, const void* q2,
                                           const void* k2, int B, int H, int NQ, int NK, int d1,
                                           int d2, float scale, int causal, int num_splits,
                                           float* kl, float* lse1, float* lse2,
                                           streamkl_stream_t stream) {
  if (num_splits < 1 || num_splits > 1024 || B < 0 || H < 0 || NQ < 0) return STREAMKL_INVALID_ARG;
  const size_t need = streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits);
  if (need > STREAMKL_STATIC_WORKSPACE_BYTES) return STREAMKL_INVALID_ARG;  // over the fixed maximum
  if (need == 0)  // no rows: nothing is computed and no device address is needed
    return streamkl_fwd_splitk(q1, k1, q2, k2, B, H, NQ, NK, d1, d2, scale, causal, num_splits,
                               nullptr, 0, kl, lse1, lse2, stream);
  void* ws = nullptr;
  const int s = static_ws_address(&ws);
  if (s != STREAMKL_OK) return s;
  // Every partial the merge reads is written by this call's first kernel,
  // so nothing in the array has to start at zero.
  return streamkl_fwd_splitk(q1, k1, q2, k2, B, H, NQ, NK, d1, d2, scale, causal, num_splits, ws,
                             STREAMKL_STATIC_WORKSPACE_BYTES, kl, lse1, lse2, stream);
}
