// Instantiations of the wide-head backward, pass 1 (dQ); see bwd_wide.cuh.
// One translation unit per pass so the build compiles them in parallel.
#include "bwd_wide.cuh"

namespace skl {

int launch_bwd_wide_pass1(const TMaps& m, int d1, int d2, const BwdArgs& a, cudaStream_t st) {
  const bool p2 = a.mode == STREAMKL_GRAD_P2;
#define SKL_WIDE_CASE(A, B) \
  if (d1 == A && d2 == B) return p2 ? launch_wide_t<A, B, 0, 1>(m, a, st) : launch_wide_t<A, B, 1, 1>(m, a, st);
  SKL_WIDE_CASE(256, 256) SKL_WIDE_CASE(256, 192) SKL_WIDE_CASE(256, 128) SKL_WIDE_CASE(256, 64)
  SKL_WIDE_CASE(256, 32) SKL_WIDE_CASE(192, 256) SKL_WIDE_CASE(192, 192) SKL_WIDE_CASE(192, 128)
  SKL_WIDE_CASE(192, 64) SKL_WIDE_CASE(192, 32) SKL_WIDE_CASE(128, 256) SKL_WIDE_CASE(128, 192)
  SKL_WIDE_CASE(64, 256) SKL_WIDE_CASE(64, 192) SKL_WIDE_CASE(32, 256) SKL_WIDE_CASE(32, 192)
#undef SKL_WIDE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace skl
