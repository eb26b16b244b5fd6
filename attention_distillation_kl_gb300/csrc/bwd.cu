// Backward kernels (in progress).
#include "kernels.cuh"
#include "ptx.cuh"

namespace skl {

int launch_bwd_fused(const TMaps&, int, int, const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
int launch_bwd_dq(const TMaps&, int, int, const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace skl
