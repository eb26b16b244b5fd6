// Forward instantiations with a head wider than 128 on either side (tile
// widths 192 and 256; the K ring then carries 64-column operand blocks).
// Kept in their own translation unit so the build compiles them in
// parallel with the narrower ones.
#include "fwd_kernel.cuh"

namespace skl {

int launch_fwd_wide(const TMaps& m, int d1, int d2, const FwdArgs& a, cudaStream_t st) {
#define SKL_FWD_CASE(A, B) \
  if (d1 == A && d2 == B) return launch_fwd_t<A, B>(m, a, st);
  SKL_FWD_CASE(256, 256) SKL_FWD_CASE(256, 192) SKL_FWD_CASE(256, 128) SKL_FWD_CASE(256, 64)
  SKL_FWD_CASE(256, 32) SKL_FWD_CASE(192, 256) SKL_FWD_CASE(192, 192) SKL_FWD_CASE(192, 128)
  SKL_FWD_CASE(192, 64) SKL_FWD_CASE(192, 32) SKL_FWD_CASE(128, 256) SKL_FWD_CASE(128, 192)
  SKL_FWD_CASE(64, 256) SKL_FWD_CASE(64, 192) SKL_FWD_CASE(32, 256) SKL_FWD_CASE(32, 192)
#undef SKL_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace skl
