// Deterministic dQ of the fused backward (grid and bound: dq_fixed_exp):
// the largest |K| of every key head, one pass over K before the fused
// launches.
#include <algorithm>

#include "bwd_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace skl {

namespace {

constexpr int kKmaxThreads = 256;

// kmax[h] = max over head h's `words` 16-byte words of k of the bf16
// magnitude bits (bits & 0x7fff order as the magnitudes do; a NaN wins),
// folded in with atomicMax, so the result does not depend on the order.
__global__ void __launch_bounds__(kKmaxThreads) kmax_kernel(const uint4* k, long long words, unsigned* kmax) {
  const uint4* p = k + size_t(blockIdx.y) * words;
  uint32_t m = 0;
  for (long long i = blockIdx.x * (long long)kKmaxThreads + threadIdx.x; i < words;
       i += (long long)gridDim.x * kKmaxThreads) {
    const uint4 w = p[i];
    const uint32_t a = max(max(w.x & 0x7fffu, (w.x >> 16) & 0x7fffu), max(w.y & 0x7fffu, (w.y >> 16) & 0x7fffu));
    const uint32_t b = max(max(w.z & 0x7fffu, (w.z >> 16) & 0x7fffu), max(w.w & 0x7fffu, (w.w >> 16) & 0x7fffu));
    m = max(m, max(a, b));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t warp_max[kKmaxThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kKmaxThreads / 32; ++w) m = max(m, warp_max[w]);
    atomicMax(kmax + blockIdx.y, m);
  }
}

}  // namespace

int launch_kmax(const void* k, int heads, long long n, int d, unsigned* kmax, cudaStream_t st) {
  if (heads <= 0 || n <= 0) return cudaSuccess;
  const long long words = n * d / 8;  // d is a multiple of 16: 8 bf16 per 16-byte word
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
  const long long per_head = (4LL * sms + heads - 1) / heads;
  const long long need = (words + kKmaxThreads - 1) / kKmaxThreads;
  dim3 grid(unsigned(std::max(1LL, std::min(per_head, std::min(need, 4096LL)))), unsigned(heads));
  kmax_kernel<<<grid, kKmaxThreads, 0, st>>>(static_cast<const uint4*>(k), words, kmax);
  return cudaGetLastError();
}

}  // namespace skl
