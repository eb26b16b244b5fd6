// Host-side launchers shared between the translation units of libstreamkl.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace skl {

constexpr int kTile = 128;  // query and key tile: 128 rows = 128 TMEM lanes

struct TMaps {
  CUtensorMap q1, k1, q2, k2;  // [BH][N][d] bf16, boxes of 64 (or 32) x 128, 128- (or 64-) byte swizzle
  CUtensorMap dq;              // [BH][NQ][dg] fp32, boxes of 16 x 32, 64-byte swizzle (both-sides backward)
  CUtensorMap dq2;             // the second side's dQ (both-sides backward)
  CUtensorMap dqw;             // [BH][NQ][dg] fp32 for the fused backward: boxes of 32 x 32 with the
                               // 128-byte swizzle when dg >= 32, else as dq (BwdArgs::dq_box says which)
};

struct FwdArgs {
  int BH, NQ, NK, causal, num_splits;
  int g1, g2;  // query heads per key head of each side (grouped key heads; 1 = one key head per query head)
  float scale1, scale2;  // S1 = scale1 Q1 K1^T, S2 = scale2 Q2 K2^T
  float* kl;
  float* lse1;
  float* lse2;
  float* partial;  // key-split partials [num_splits][5][BH*NQ], or null
  int* status;
  // CTA order: heads in groups of head_group whose query tiles interleave,
  // longest first (causal), so the long CTAs of every head in a group start
  // early; groups follow one another (1 = head after head).  The group is
  // sized so that its heads' re-read operands stay in L2 (head_group_for).
  int head_group = 1;
};

struct BwdArgs {
  int BH, NQ, NK, causal, mode;
  int dg;  // the gradient side's head dim: row length of dq, dk (at most the kernel's tile width)
  int g1, g2;  // query heads per key head of each side; dk has BH / g_grad heads
  // Query heads of the wide-head dK pass: -1 = every head (grid.y = BH);
  // j >= 0 = head j of every key-head group only (grid.y = BH / g_grad), dK
  // stored (j = 0) or added in place (j > 0), so launches j = 0, 1, ... sum
  // in a fixed order.  (The fused kernel always takes every head.)
  int hsel;
  float scale1, scale2;
  const float* kl;
  const float* lse1;
  const float* lse2;
  const float* dkl;
  float* dq;  // fp32 [BH][NQ][dg]
  float* dk;  // fp32 [BH][NK][dg]
  int* status;
  float* dq2;    // both-sides backward: dQ2, dK2 (dq, dk then hold dQ1, dK1)
  float* dk2;
  int dq_box;    // fused backward: width of the dQ reduce-add boxes, 32 (dqw, 128-byte swizzle) or 16
  // Fused backward, deterministic mode: every dQ contribution rounded to its
  // row's grid (dq_fixed_exp) so the fp32 sums are exact in any order.
  // kmax: per key head of the gradient side, the largest |K| as bf16
  // magnitude bits (launch_kmax); the both-sides kernel reads side 1's at
  // [0, BH) and side 2's at [BH, 2 BH).
  int dq_fixed;
  const unsigned* kmax;
  // Deterministic mode with grouped key heads, one launch for all query
  // heads (all null otherwise): ticket (zeroed) hands out the CTAs' units
  // (key tile, query head) in launch order; dk_turns [B * HK_g][key tiles]
  // (zeroed) counts the query heads of a group that have added their dK to
  // a key tile, which they do in head order; dk_abort (zeroed) is set by a
  // CTA that gave up, so the later heads do not wait for it.
  int* ticket;
  int* dk_turns;
  int* dk_abort;
  // CTA order of the fused backward, as FwdArgs::head_group (key tiles
  // instead of query tiles; 1 whenever ticket is set).
  int head_group = 1;
};

// Unit u of a launch over BH heads x n tiles, heads in groups of G whose
// tiles interleave: (head, tile index).  A bijection of [0, BH n).
__host__ __device__ inline void grouped_unit(int u, int BH, int n, int G, int& head, int& tile) {
  const int g0 = u / (G * n) * G;       // first head of u's group
  const int gs = BH - g0 < G ? BH - g0 : G;  // heads in that group
  const int r = u - g0 * n;             // in [0, gs n)
  tile = r / gs;
  head = g0 + r % gs;
}

// Each returns a cudaError_t value (cudaSuccess = 0).  d1, d2 and d are the
// kernels' tile widths (32, 64, 128, 192 or 256): a head dim below its tile width is
// read with the columns past it zero-filled by the TMA.
int launch_fwd(const TMaps& m, int d1, int d2, const FwdArgs& a, cudaStream_t st);
int launch_fwd_wide(const TMaps& m, int d1, int d2, const FwdArgs& a, cudaStream_t st);  // a side above 128
int launch_splitk_reduce(const float* partial, int rows, int num_splits, float* kl, float* lse1,
                         float* lse2, cudaStream_t st);
int launch_bwd_fused(const TMaps& m, int d1, int d2, const BwdArgs& a, cudaStream_t st);
// Deterministic dQ: kmax[h] = bits of max |k| over head h of k ([heads][n][d]
// bf16), into a zeroed kmax.
int launch_kmax(const void* k, int heads, long long n, int d, unsigned* kmax, cudaStream_t st);
int launch_bwd_both(const TMaps& m, int d, const BwdArgs& a, cudaStream_t st);  // d1 = d2 = d, 32 or 64
// Backward with a side above 128: pass 0 writes dK (ordered launches over a
// key-head group via hsel), pass 1 writes dQ; neither uses atomics.
int launch_bwd_wide_pass0(const TMaps& m, int d1, int d2, const BwdArgs& a, cudaStream_t st);
int launch_bwd_wide_pass1(const TMaps& m, int d1, int d2, const BwdArgs& a, cudaStream_t st);
int launch_ex2_probe(float* out, int blocks, int iters, cudaStream_t st);
int launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t st);
int launch_turn_selftest(int* words, int* status, uint64_t limit_ns, cudaStream_t st);

}  // namespace skl
