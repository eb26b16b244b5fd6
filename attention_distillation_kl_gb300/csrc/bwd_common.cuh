// Device helpers shared by the backward kernels: bf16 packing, swizzled
// shared-memory row stores and the per-element dS formula of both modes.
#pragma once

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace skl {

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Writes one 128-element bf16 row (64 packed registers) of a [rows][128]
// operand in the 128-byte-swizzled layout: two 64-column blocks of
// [rows][128 B], 16-byte chunk c of row r stored at chunk c ^ (r % 8).
__device__ __forceinline__ void store_row_sw128(uint32_t base, int r, const uint32_t (&v)[64]) {
  const uint32_t rb = base + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int c16 = 0; c16 < 16; ++c16) {
    const int blk = c16 >> 3, c = c16 & 7;
    st_shared_v4(rb + blk * (kTile * 128) + ((c ^ (r & 7)) << 4), v[4 * c16], v[4 * c16 + 1],
                 v[4 * c16 + 2], v[4 * c16 + 3]);
  }
}

// Writes one 64-element half (block `blk`) of such a row from 32 packed registers.
__device__ __forceinline__ void store_half_row_sw128(uint32_t base, int r, int blk, const uint32_t (&v)[32]) {
  const uint32_t rb = base + blk * (kTile * 128) + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st_shared_v4(rb + ((c ^ (r & 7)) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// dS for 32 consecutive query columns of one key row (thread), packed to
// bf16 pairs.  pa/pb/pw: per-column parameters in shared memory:
//   mode P2: pa = -LSE1 log2e, pb = -LSE2 log2e, pw = s dKL
//   mode P1: pa = -LSE1 log2e, pb = -(LSE1 - LSE2 + KL), pw = s dKL
// (the softmax scale s rides on dS, so dK = dS^T Q and dQ = dS K need no
// further scaling)
// Columns < first_visible (causal) or all columns when the key is past NK
// (first_visible > 128) give 0.
template <int MODE, bool kMask>
__device__ __forceinline__ void ds_chunk(const uint32_t (&x1u)[32], const uint32_t (&x2u)[32],
                                         const float* pa, const float* pb, const float* pw, float c,
                                         float s, int col0, int first_visible, uint32_t* out16) {
  const uint64_t C = f2(c, c), S = f2(s, s);
#pragma unroll
  for (int k = 0; k < 32; k += 4) {
    const float4 A = *reinterpret_cast<const float4*>(pa + col0 + k);
    const float4 Bv = *reinterpret_cast<const float4*>(pb + col0 + k);
    const float4 W = *reinterpret_cast<const float4*>(pw + col0 + k);
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const uint64_t X1 = f2(__uint_as_float(x1u[k + e]), __uint_as_float(x1u[k + e + 1]));
      const uint64_t X2 = f2(__uint_as_float(x2u[k + e]), __uint_as_float(x2u[k + e + 1]));
      const uint64_t AA = e == 0 ? f2(A.x, A.y) : f2(A.z, A.w);
      const uint64_t BB = e == 0 ? f2(Bv.x, Bv.y) : f2(Bv.z, Bv.w);
      const uint64_t WW = e == 0 ? f2(W.x, W.y) : f2(W.z, W.w);
      float ea, eb;
      f2_split(f2_fma(X1, C, AA), ea, eb);
      const uint64_t P1 = f2(ex2(ea), ex2(eb));
      uint64_t D;
      if (MODE == STREAMKL_GRAD_P2) {
        f2_split(f2_fma(X2, C, BB), ea, eb);
        D = f2_mul(WW, f2_sub(f2(ex2(ea), ex2(eb)), P1));
      } else {
        D = f2_mul(f2_mul(WW, P1), f2_fma(f2_sub(X1, X2), S, BB));
      }
      float da, db;
      f2_split(D, da, db);
      if (kMask) {
        if (col0 + k + e < first_visible) da = 0.f;
        if (col0 + k + e + 1 < first_visible) db = 0.f;
      }
      out16[(k + e) / 2] = pack_bf16(da, db);
    }
  }
}

}  // namespace skl
