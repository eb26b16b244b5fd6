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

// How a dK row chunk reaches global memory: plain store (the CTA owns the
// key head), atomic add (several CTAs of a key-head group at once) or
// read-add-write (the launches of a group run one after the other).
// (The read in the read-add-write bypasses L1: within one launch the
// previous value may have been written from another SM.)
enum { kDkStore = 0, kDkAtomic = 1, kDkAdd = 2 };

__device__ __forceinline__ void put_dk4(float* p, float4 v, int how) {
  float4* q = reinterpret_cast<float4*>(p);
  if (how == kDkStore) {
    *q = v;
  } else if (how == kDkAtomic) {
    atomicAdd(q, v);
  } else {
    const float4 o = __ldcg(q);
    *q = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
  }
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

// dS for 32 consecutive key columns of one query row (thread), packed to
// bf16 pairs.  Per-row parameters, each broadcast to both halves of a pair:
//   mode P2: NA = -LSE1 log2e, NB = -LSE2 log2e, WW = s2 dKL
//   mode P1: NA = -LSE1 log2e, NB = -(LSE1 - LSE2 + KL), WW = s1 dKL
// and per-launch constants C1 = s1 log2e, C2 = s2 log2e, S1 = s1,
// NR = -s2 / s1 (the gradient side's softmax scale rides on dS, so
// dK = dS^T Q and dQ = dS K need no further scaling; in mode P1 the
// log-ratio S1 - S2 - LSE1 + LSE2 is s1 (x1 - (s2/s1) x2) + LSE2 - LSE1).
// Columns k > lim_rel (causal, or past NK) give 0.  A row past NQ has
// NA = -inf (and NB = -inf in mode P2, WW = 0), so every product is an exact 0.
template <int MODE, bool kMask>
__device__ __forceinline__ void ds_chunk_row(const uint32_t (&x1u)[32], const uint32_t (&x2u)[32],
                                             uint64_t C1, uint64_t C2, uint64_t S1, uint64_t NR, uint64_t NA,
                                             uint64_t NB, uint64_t WW, int lim_rel, uint32_t* out16) {
#pragma unroll
  for (int k = 0; k < 32; k += 2) {
    const uint64_t X1 = f2(__uint_as_float(x1u[k]), __uint_as_float(x1u[k + 1]));
    const uint64_t X2 = f2(__uint_as_float(x2u[k]), __uint_as_float(x2u[k + 1]));
    float ea, eb;
    f2_split(f2_fma(X1, C1, NA), ea, eb);
    const uint64_t P1 = f2(ex2(ea), ex2(eb));
    uint64_t D;
    if (MODE == STREAMKL_GRAD_P2) {
      f2_split(f2_fma(X2, C2, NB), ea, eb);
      D = f2_mul(WW, f2_sub(f2(ex2(ea), ex2(eb)), P1));
    } else {
      D = f2_mul(f2_mul(WW, P1), f2_fma(f2_fma(X2, NR, X1), S1, NB));
    }
    float da, db;
    f2_split(D, da, db);
    if (kMask) {
      if (k > lim_rel) da = 0.f;
      if (k + 1 > lim_rel) db = 0.f;
    }
    out16[k / 2] = pack_bf16(da, db);
  }
}

// Writes 32 bf16 columns [col, col + 32) (col a multiple of 32) of row r of
// such an operand from 16 packed registers.
__device__ __forceinline__ void store_cols32_sw128(uint32_t base, int r, int col, const uint32_t (&v)[16]) {
  const uint32_t rb = base + (col >> 6) * (kTile * 128) + (r >> 3) * 1024 + (r & 7) * 128;
  const int c0 = (col & 63) >> 3;  // first 16-byte chunk of the 32 columns
#pragma unroll
  for (int k = 0; k < 4; ++k)
    st_shared_v4(rb + (((c0 + k) ^ (r & 7)) << 4), v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

// Both gradient sides from one pair of exponentials: for 32 key columns of
// one query row, dS2 = s2 dKL (P2 - P1) into out2 and dS1 = s1 dKL P1 (r - KL)
// into out1 (packed bf16 pairs).  Per-row parameters as in ds_chunk_row:
// NA = -LSE1 log2e, NB2 = -LSE2 log2e, NB1 = -(LSE1 - LSE2 + KL),
// W2 = s2 dKL, W1 = s1 dKL; constants C1, C2, S1, NR as there.
template <bool kMask>
__device__ __forceinline__ void ds_chunk_row_both(const uint32_t (&x1u)[32], const uint32_t (&x2u)[32],
                                                  uint64_t C1, uint64_t C2, uint64_t S1, uint64_t NR,
                                                  uint64_t NA, uint64_t NB2, uint64_t NB1, uint64_t W2,
                                                  uint64_t W1, int lim_rel, uint32_t (&out1)[16],
                                                  uint32_t (&out2)[16]) {
#pragma unroll
  for (int k = 0; k < 32; k += 2) {
    const uint64_t X1 = f2(__uint_as_float(x1u[k]), __uint_as_float(x1u[k + 1]));
    const uint64_t X2 = f2(__uint_as_float(x2u[k]), __uint_as_float(x2u[k + 1]));
    float ea, eb;
    f2_split(f2_fma(X1, C1, NA), ea, eb);
    const uint64_t P1 = f2(ex2(ea), ex2(eb));
    f2_split(f2_fma(X2, C2, NB2), ea, eb);
    const uint64_t D2 = f2_mul(W2, f2_sub(f2(ex2(ea), ex2(eb)), P1));
    const uint64_t D1 = f2_mul(f2_mul(W1, P1), f2_fma(f2_fma(X2, NR, X1), S1, NB1));
    float a1, b1, a2, b2;
    f2_split(D1, a1, b1);
    f2_split(D2, a2, b2);
    if (kMask) {
      if (k > lim_rel) a1 = a2 = 0.f;
      if (k + 1 > lim_rel) b1 = b2 = 0.f;
    }
    out1[k / 2] = pack_bf16(a1, b1);
    out2[k / 2] = pack_bf16(a2, b2);
  }
}

// Deterministic dQ: every contribution to a dQ row is rounded to a grid of
// 2^-e (e per query row) before its fp32 reduce-add.  A sum of multiples of
// 2^-e is exact in fp32 while it stays below 2^24 grid steps, so the sums
// come out the same whatever order the reduce-adds land in.  e comes from a
// bound on |dQ_id| that holds for every partial sum of the row:
//   |dQ_id| <= s |dKL_i| kmax C_i,  kmax = max |K_g| of the key head,
//   C_i = sum_k |dS_ik| / |dKL_i|, with TV_i = sum_k max(P2 - P1, 0)
//        <= min(1, sqrt(KL_i / 2)) (Pinsker):
//     mode P2: sum_k |P2_ik - P1_ik| = 2 TV_i;
//     mode P1: sum_k P1_ik |r_ik - KL_i| <= 2 KL_i + 2 TV_i
//              (r = ln P1 - ln P2; E_P1 |r| = KL + 2 E_P1[max(-r, 0)] and
//              E_P1[max(ln(P2/P1), 0)] <= sum max(P2 - P1, 0) = TV).
// KL_i is the forward's value; the bound adds slack for its rounding, for
// the recomputed probabilities and for the bf16 rounding of dS.  2^e times
// the bound stays at or below 2^22, so one contribution is rounded by the
// addend 1.5 * 2^(23 - e) (which holds it in the binade whose step is 2^-e)
// to within 2^-22 of the bound, and partial sums keep a factor of 4 below
// 2^24 steps: a bound off by less than that costs nothing; one off by more
// rounds its contributions coarser, still on the grid.
__device__ __forceinline__ int dq_fixed_exp(int mode, float sg, float dkl, float kl, float kmax) {
  // explicitly rounded operations: every CTA that adds to a row must reach
  // the same e for it, whatever the compiler contracts elsewhere
  const float k = __fadd_rn(fmaxf(kl, 0.f), 1.0e-4f);
  const float tv = __fadd_rn(fminf(1.f, __fsqrt_rn(__fmul_rn(k, 0.5f))), 1.0e-4f);
  const float c = mode == STREAMKL_GRAD_P2 ? __fmul_rn(2.f, tv) : __fmul_rn(2.f, __fadd_rn(k, tv));
  const float bound = __fmul_rn(__fmul_rn(__fmul_rn(__fmul_rn(sg, fabsf(dkl)), kmax), c), 1.0078125f);
  if (!(bound > 0.f && bound <= 3.0e38f)) return 0;  // zero (nothing to add) or not finite
  const int E = int((__float_as_uint(bound) >> 23) & 255u);  // bound < 2^(E - 126)
  // 2^e bound <= 2^22, with e at most 126: every nonzero grid value is then a
  // normal float (no flushing of subnormals can enter a sum), and rows whose
  // bound is below 2^-104 keep a grid of 2^-126
  return max(-100, min(126, 148 - E));
}

// 2^e as a float, for |e| <= 126.
__device__ __forceinline__ float exp2_int(int e) { return __uint_as_float(uint32_t(e + 127) << 23); }

}  // namespace skl
