// The forward kernel template (shared by the translation units that
// instantiate it for each pair of tile widths).
//
// Forward kernel: one CTA streams all visible key tiles past one 128-row query
// tile and keeps the coupled online statistics of the StreamKL article
// ("Online formula", "Forward") in registers:
//   m1, m2   running maxima of the raw logits q.k
//   l1, l2   running sums of 2^(c (x - m))        (c = s log2 e of that side)
//   acc      running sum of 2^(c1 (x1 - m1)) (x1 - rho x2),  rho = s2 / s1
// When m1 moves, l1 and acc are multiplied by 2^(c1 (m1_old - m1_new)) -- a
// vector rescale per row, never a B_Q x d matrix.  At the end
//   LSE = s m + ln l,  KL = s1 acc / l1 + LSE2 - LSE1
// (s1 (x1 - rho x2) = S1 - S2, so s1 acc / l1 is the P1-weighted mean of
// S1 - S2).
//
// GB300 mapping (one CTA per SM):
//   TMA producer warp: Q1/Q2 once, then K1_j/K2_j (key head h / G) into a ring
//   MMA warp: TMEM owner and MMA issuer: S1 = Q1 K1_j^T and S2 = Q2 K2_j^T
//               (tcgen05, M = N = 128, bf16 -> fp32) into one of two TMEM
//               buffers of 256 columns, so tile j+1 is multiplied while the
//               statistics of tile j are reduced.  The whole warp runs the
//               loop and one elected lane issues (see elect_one).
//   statistics warps (the first 4 x FwdLayout::kWGs): thread = query row
//               (TMEM lane); warpgroup w takes key columns [w kCols, (w+1)
//               kCols) of every tile, and the partial states are merged at
//               the end with the same algebra as the key-split reduce.  Four
//               warpgroups of 32 columns (four warps per SM sub-partition)
//               hide the latency of the ex2 and FMA chains better than two
//               of 64; the loop is close to the issue and ex2 limits.
// Head dims above 128 (tile widths 192, 256): the K ring carries 64-column
// operand blocks instead of whole key tiles (see FwdLayout); the MMA warp
// multiplies each block as it lands.
// With num_splits > 1 (article section "GPU kernel engineering", split-K) a
// CTA covers only its share of the key tiles and writes (m1, l1, acc, m2, l2)
// instead of the final values; splitk_reduce_kernel merges them.
#pragma once

#include "kernels.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace skl {

// Shared memory: Q1, Q2 resident, then the K ring.  Up to tile width 128 on
// both sides a ring stage holds a whole key tile (K1 and K2); wider heads
// (192, 256) leave no room for two such stages next to Q, so the ring then
// carries one operand block (64 columns of one side, at most 16 KB) per
// slot and a key tile passes through it as D1/64 + D2/64 blocks.
template <int D1, int D2>
struct FwdLayout {
  static constexpr bool kRing = D1 > 128 || D2 > 128;
  // Statistics warpgroups: each takes kCols key columns of every tile.  Up
  // to tile width 128, four warpgroups of one 32-column chunk each (four
  // statistics warps per SM sub-partition to hide the latency of the ex2
  // and FMA chains, 96 registers a thread); with the block ring, whose MMA
  // warp issues block by block and is slowed by more warps beside it, two
  // warpgroups of 64 columns.  Then one producer warp and one MMA warp.
  static constexpr int kWGs = kRing ? 2 : 4;
  static constexpr int kStatWarps = 4 * kWGs;
  static constexpr int kCols = kTile / kWGs;
  static constexpr int kProdWarp = kStatWarps, kMmaWarp = kStatWarps + 1;
  static constexpr int kThreads = 32 * (kStatWarps + 2);
  static constexpr uint32_t kQ1 = kTile * D1 * 2, kQ2 = kTile * D2 * 2;
  static constexpr uint32_t kK1 = kTile * D1 * 2, kK2 = kTile * D2 * 2;
  static constexpr int kNb1 = OpTile<D1>::kBlocks, kNb2 = OpTile<D2>::kBlocks;  // ring blocks per key tile
  static constexpr uint32_t kStage = kRing ? 16384u : kK1 + kK2;
  static constexpr int kStagesFit = int((210u * 1024u - kQ1 - kQ2) / kStage);
  static constexpr int kStages = kRing ? (kStagesFit > 8 ? 8 : kStagesFit) : (kStagesFit > 4 ? 4 : kStagesFit);
  static constexpr uint32_t oQ1 = 0, oQ2 = kQ1, oK = kQ1 + kQ2;
  static constexpr uint32_t oBar = oK + kStages * kStage;
  // q_full, k_full[S], k_empty[S], s_full[2], s_empty[2], mma_done
  static constexpr int kNumBars = 1 + 2 * kStages + 4 + 1;
  static constexpr uint32_t oMisc = oBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr uint32_t oMerge = (oMisc + 8 + 15) / 16 * 16;
  static constexpr uint32_t kBytes = oMerge + (kWGs - 1) * kTile * 5 * 4;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static_assert(kStages >= 2, "shared memory ring needs two stages");
  static_assert(kAlloc <= 232448, "over the 227 KB shared memory limit");
};

// Per-row running state of one thread.
struct RowStats {
  float m1, m2, l1, l2, acc;
};

// The sums of one 32-column chunk against the reference nb = -c m of each
// side: l1 = sum 2^(c1 x1 + nb1), l2 = sum 2^(c2 x2 + nb2) and
// acc = sum 2^(c1 x1 + nb1) (x1 - rho x2), columns past lim_rel masked.
// c1, c2: s log2 e of each side; NR = -s2 / s1 in both lanes (x1 - rho x2 is
// one fma, exactly x1 - x2 when the scales are equal).  Pairs of columns go
// through the packed FP32 pipe, in two chains (pairs k, k + 1 and k + 2,
// k + 3) for instruction-level parallelism.  Taken against the running
// maxima as they stand (the fast path, no maximum pass and no rescale),
// the sums are exact as long as no term overflows: the online recurrence
// holds for any reference at or above the values seen so far, and fp32
// keeps its relative precision at any scale.
template <bool kMask>
__device__ __forceinline__ void chunk_sums(const uint32_t (&x1)[32], const uint32_t (&x2)[32], uint64_t C1,
                                           uint64_t C2, uint64_t NR, uint64_t NB1, uint64_t NB2, int lim_rel,
                                           float& l1, float& l2, float& acc) {
  uint64_t L1a = f2(0.f, 0.f), L2a = L1a, ACa = L1a, L1b = L1a, L2b = L1a, ACb = L1a;
#pragma unroll
  for (int k = 0; k < 32; k += 4) {
    const uint64_t XA1 = f2(__uint_as_float(x1[k]), __uint_as_float(x1[k + 1]));
    const uint64_t XA2 = f2(__uint_as_float(x2[k]), __uint_as_float(x2[k + 1]));
    const uint64_t XB1 = f2(__uint_as_float(x1[k + 2]), __uint_as_float(x1[k + 3]));
    const uint64_t XB2 = f2(__uint_as_float(x2[k + 2]), __uint_as_float(x2[k + 3]));
    float e1a, e1b, e2a, e2b, g1a, g1b, g2a, g2b;
    f2_split(f2_fma(XA1, C1, NB1), e1a, e1b);
    f2_split(f2_fma(XA2, C2, NB2), e2a, e2b);
    f2_split(f2_fma(XB1, C1, NB1), g1a, g1b);
    f2_split(f2_fma(XB2, C2, NB2), g2a, g2b);
    float p1a = ex2(e1a), p1b = ex2(e1b), p2a = ex2(e2a), p2b = ex2(e2b);
    float q1a = ex2(g1a), q1b = ex2(g1b), q2a = ex2(g2a), q2b = ex2(g2b);
    if (kMask) {
      if (k > lim_rel) { p1a = 0.f; p2a = 0.f; }
      if (k + 1 > lim_rel) { p1b = 0.f; p2b = 0.f; }
      if (k + 2 > lim_rel) { q1a = 0.f; q2a = 0.f; }
      if (k + 3 > lim_rel) { q1b = 0.f; q2b = 0.f; }
    }
    const uint64_t P1 = f2(p1a, p1b), Q1 = f2(q1a, q1b);
    L1a = f2_add(L1a, P1);
    L2a = f2_add(L2a, f2(p2a, p2b));
    ACa = f2_fma(P1, f2_fma(XA2, NR, XA1), ACa);
    L1b = f2_add(L1b, Q1);
    L2b = f2_add(L2b, f2(q2a, q2b));
    ACb = f2_fma(Q1, f2_fma(XB2, NR, XB1), ACb);
  }
  float u, v;
  f2_split(f2_add(L1a, L1b), u, v);
  l1 = u + v;
  f2_split(f2_add(L2a, L2b), u, v);
  l2 = u + v;
  f2_split(f2_add(ACa, ACb), u, v);
  acc = u + v;
}

// Folds one 32-column chunk into the running state exactly: the maxima move
// to the chunk's, the state is rescaled once, and the chunk's sums are taken
// against the new maxima.  Masked columns (k > lim_rel) move nothing.
template <bool kMask>
__device__ __forceinline__ void fold_one(RowStats& st, const uint32_t (&x1)[32], const uint32_t (&x2)[32],
                                         uint64_t C1, uint64_t C2, uint64_t NR, float c1, float c2,
                                         int lim_rel) {
  float ta1 = st.m1, ta2 = st.m2, tb1 = kNegBig, tb2 = kNegBig;
#pragma unroll
  for (int k = 0; k < 32; k += 4) {
    const bool o0 = !kMask || k <= lim_rel, o1 = !kMask || k + 1 <= lim_rel;
    const bool o2 = !kMask || k + 2 <= lim_rel, o3 = !kMask || k + 3 <= lim_rel;
    ta1 = max3(ta1, o0 ? __uint_as_float(x1[k]) : kNegBig, o1 ? __uint_as_float(x1[k + 1]) : kNegBig);
    ta2 = max3(ta2, o0 ? __uint_as_float(x2[k]) : kNegBig, o1 ? __uint_as_float(x2[k + 1]) : kNegBig);
    tb1 = max3(tb1, o2 ? __uint_as_float(x1[k + 2]) : kNegBig, o3 ? __uint_as_float(x1[k + 3]) : kNegBig);
    tb2 = max3(tb2, o2 ? __uint_as_float(x2[k + 2]) : kNegBig, o3 ? __uint_as_float(x2[k + 3]) : kNegBig);
  }
  const float t1 = fmaxf(ta1, tb1), t2 = fmaxf(ta2, tb2);
  const float a1 = ex2((st.m1 - t1) * c1);
  const float a2 = ex2((st.m2 - t2) * c2);
  st.m1 = t1;
  st.m2 = t2;
  const float nb1 = -t1 * c1, nb2 = -t2 * c2;
  float l1, l2, acc;
  chunk_sums<kMask>(x1, x2, C1, C2, NR, f2(nb1, nb1), f2(nb2, nb2), lim_rel, l1, l2, acc);
  st.l1 = fmaf(st.l1, a1, l1);
  st.acc = fmaf(st.acc, a1, acc);
  st.l2 = fmaf(st.l2, a2, l2);
}

// Folds 64 consecutive key columns (two 32-column chunks) into the running
// state exactly: the maxima move to the columns', the state is rescaled
// once, and the chunks' sums are taken against the new maxima.  Columns k
// with k > lim_rel (relative to the first chunk; causal, or past NK) are
// masked: they neither move the maxima nor add to the sums.
template <bool kMask>
__device__ __forceinline__ void fold_pair(RowStats& st, const uint32_t (&xa1)[32], const uint32_t (&xa2)[32],
                                          const uint32_t (&xb1)[32], const uint32_t (&xb2)[32], uint64_t C1,
                                          uint64_t C2, uint64_t NR, float c1, float c2, int lim_rel) {
  float ta1 = st.m1, ta2 = st.m2, tb1 = kNegBig, tb2 = kNegBig;
#pragma unroll
  for (int k = 0; k < 32; k += 2) {
    const bool oa = !kMask || k <= lim_rel, ob = !kMask || k + 1 <= lim_rel;
    const bool pa = !kMask || k + 32 <= lim_rel, pb = !kMask || k + 33 <= lim_rel;
    ta1 = max3(ta1, oa ? __uint_as_float(xa1[k]) : kNegBig, ob ? __uint_as_float(xa1[k + 1]) : kNegBig);
    ta2 = max3(ta2, oa ? __uint_as_float(xa2[k]) : kNegBig, ob ? __uint_as_float(xa2[k + 1]) : kNegBig);
    tb1 = max3(tb1, pa ? __uint_as_float(xb1[k]) : kNegBig, pb ? __uint_as_float(xb1[k + 1]) : kNegBig);
    tb2 = max3(tb2, pa ? __uint_as_float(xb2[k]) : kNegBig, pb ? __uint_as_float(xb2[k + 1]) : kNegBig);
  }
  const float t1 = fmaxf(ta1, tb1), t2 = fmaxf(ta2, tb2);
  const float a1 = ex2((st.m1 - t1) * c1);
  const float a2 = ex2((st.m2 - t2) * c2);
  st.m1 = t1;
  st.m2 = t2;
  const float nb1 = -t1 * c1, nb2 = -t2 * c2;
  const uint64_t NB1 = f2(nb1, nb1), NB2 = f2(nb2, nb2);
  float l1a, l2a, aca, l1b, l2b, acb;
  chunk_sums<kMask>(xa1, xa2, C1, C2, NR, NB1, NB2, lim_rel, l1a, l2a, aca);
  chunk_sums<kMask>(xb1, xb2, C1, C2, NR, NB1, NB2, lim_rel - 32, l1b, l2b, acb);
  st.l1 = fmaf(st.l1, a1, l1a + l1b);
  st.acc = fmaf(st.acc, a1, aca + acb);
  st.l2 = fmaf(st.l2, a2, l2a + l2b);
}

// Fast path of fold_pair: the 64 columns exponentiated against the running
// maxima as they stand, with no maximum pass and no rescale (see chunk_sums
// for why that is exact).  Returns false -- the state untouched -- when a
// partial sum reaches 2^64 (a logit above the reference by more than 64 / c,
// the first tile of a row whose reference is still kNegBig, or a non-finite
// input): the caller then folds the tile exactly with fold_pair.
template <bool kMask>
__device__ __forceinline__ bool fold_pair_fast(RowStats& st, const uint32_t (&xa1)[32], const uint32_t (&xa2)[32],
                                               const uint32_t (&xb1)[32], const uint32_t (&xb2)[32], uint64_t C1,
                                               uint64_t C2, uint64_t NR, float c1, float c2, int lim_rel) {
  const float nb1 = -st.m1 * c1, nb2 = -st.m2 * c2;
  const uint64_t NB1 = f2(nb1, nb1), NB2 = f2(nb2, nb2);
  float l1a, l2a, aca, l1b, l2b, acb;
  chunk_sums<kMask>(xa1, xa2, C1, C2, NR, NB1, NB2, lim_rel, l1a, l2a, aca);
  chunk_sums<kMask>(xb1, xb2, C1, C2, NR, NB1, NB2, lim_rel - 32, l1b, l2b, acb);
  const float l1 = l1a + l1b, l2 = l2a + l2b;
  if (!(l1 < 18446744073709551616.f && l2 < 18446744073709551616.f)) return false;  // 2^64
  st.l1 += l1;
  st.acc += aca + acb;
  st.l2 += l2;
  return true;
}

template <int D1, int D2>
__global__ void __launch_bounds__(FwdLayout<D1, D2>::kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq1, const __grid_constant__ CUtensorMap tk1,
               const __grid_constant__ CUtensorMap tq2, const __grid_constant__ CUtensorMap tk2,
               const FwdArgs a) {
  using L = FwdLayout<D1, D2>;
  using T1 = OpTile<D1>;
  using T2 = OpTile<D2>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int nqt = (a.NQ + kTile - 1) / kTile;
  int bh, t;
  grouped_unit(int(blockIdx.y) * int(gridDim.x) + int(blockIdx.x), a.BH, nqt, a.head_group, bh, t);
  const int qt = a.causal ? (nqt - 1 - t) : t;  // longest rows first
  const int split = blockIdx.z;
  const int q0 = qt * kTile;
  const int off = a.NK - a.NQ;
  const int kend = a.causal ? min(q0 + kTile, a.NQ) + off : a.NK;
  const int nkt_all = (kend + kTile - 1) / kTile;
  const int kt_lo = int((long long)split * nkt_all / a.num_splits);
  const int kt_hi = int((long long)(split + 1) * nkt_all / a.num_splits);
  const int nkt = kt_hi - kt_lo;

  const uint32_t bar0 = sb + L::oBar;
  const uint32_t bar_q = bar0;
  auto bar_kfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_kempty = [&](int s) { return bar0 + 8u * (1 + L::kStages + s); };
  auto bar_sfull = [&](int b) { return bar0 + 8u * (1 + 2 * L::kStages + b); };
  auto bar_sempty = [&](int b) { return bar0 + 8u * (3 + 2 * L::kStages + b); };
  const uint32_t bar_done = bar0 + 8u * (5 + 2 * L::kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oMisc + 4);
  const Ctl ctl{abort_flag, a.status};

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_sfull(b), 1);
      mbar_init(bar_sempty(b), L::kStatWarps);
    }
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == L::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == L::kProdWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && nkt > 0) {
      tma_prefetch_desc(&tq1);
      tma_prefetch_desc(&tk1);
      tma_prefetch_desc(&tq2);
      tma_prefetch_desc(&tk2);
      mbar_arrive_expect_tx(bar_q, L::kQ1 + L::kQ2);
      T1::load(sb + L::oQ1, &tq1, bar_q, q0, bh);
      T2::load(sb + L::oQ2, &tq2, bar_q, q0, bh);
      int issued = 0;  // ring fills issued (key tiles, or blocks with the block ring)
      if constexpr (L::kRing) {
        bool go = true;
        for (int j = 0; j < nkt && go; ++j) {
          const int k0 = (kt_lo + j) * kTile;
#pragma unroll 1
          for (int b = 0; b < L::kNb1 + L::kNb2; ++b) {
            const int u = j * (L::kNb1 + L::kNb2) + b, s = u % L::kStages;
            if (!mbar_wait(bar_kempty(s), ((u / L::kStages) & 1) ^ 1, ctl)) {
              go = false;
              break;
            }
            const uint32_t st = sb + L::oK + s * L::kStage;
            if (!SKL_CHECK(a.status, s < L::kStages && k0 < a.NK + kTile)) {
              go = false;
              break;
            }
            if (b < L::kNb1) {
              mbar_arrive_expect_tx(bar_kfull(s), T1::kBlockBytes);
              tma_load_3d(st, &tk1, bar_kfull(s), b * T1::kBox, k0, bh / a.g1);
            } else {
              mbar_arrive_expect_tx(bar_kfull(s), T2::kBlockBytes);
              tma_load_3d(st, &tk2, bar_kfull(s), (b - L::kNb1) * T2::kBox, k0, bh / a.g2);
            }
            issued = u + 1;
          }
        }
      } else {
        for (int j = 0; j < nkt; ++j) {
          const int s = j % L::kStages;
          const uint32_t ph = (j / L::kStages) & 1;
          if (!mbar_wait(bar_kempty(s), ph ^ 1, ctl)) break;
          mbar_arrive_expect_tx(bar_kfull(s), L::kStage);
          const int k0 = (kt_lo + j) * kTile;
          const uint32_t st = sb + L::oK + s * L::kStage;
          T1::load(st, &tk1, bar_kfull(s), k0, bh / a.g1);
          T2::load(st + L::kK1, &tk2, bar_kfull(s), k0, bh / a.g2);
          issued = j + 1;
        }
      }
      if (*abort_flag) {  // let the copies already started land before the CTA exits
        mbar_drain(bar_q, 0, 200000000ull);
        for (int j = issued > L::kStages ? issued - L::kStages : 0; j < issued; ++j)
          mbar_drain(bar_kfull(j % L::kStages), (j / L::kStages) & 1, 200000000ull);  // (ring fills)
      }
    }
  } else if (warp == L::kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // (the whole warp runs the loop; the elected lane issues)
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
    if (nkt > 0 && mbar_wait_warp(bar_q, 0, ctl)) {
      for (int j = 0; j < nkt; ++j) {
        const int b = j & 1;
        const uint32_t bph = (j >> 1) & 1;
        const uint32_t d1 = tmem + b * 256, d2 = d1 + 128;
        if constexpr (L::kRing) {
          // one ring block at a time: its K steps against the resident Q
          if (!mbar_wait_warp(bar_sempty(b), bph ^ 1, ctl)) break;
          bool go = true;
#pragma unroll 1
          for (int blk = 0; blk < L::kNb1 + L::kNb2; ++blk) {
            const int u = j * (L::kNb1 + L::kNb2) + blk, s = u % L::kStages;
            if (!mbar_wait_warp(bar_kfull(s), (u / L::kStages) & 1, ctl)) {
              go = false;
              break;
            }
            tc_fence_after();
            const uint32_t ks = sb + L::oK + s * L::kStage;
            if (blk < L::kNb1) {
              constexpr int kSteps = T1::kBox / 16;
#pragma unroll
              for (int jj = 0; jj < kSteps; ++jj) {
                const int kk = blk * kSteps + jj;
                mma_bf16_ss(leader, d1, T1::desc_k(sb + L::oQ1 + T1::off_k(kk)), T1::desc_k(ks + jj * 32), idesc,
                            kk > 0);
              }
            } else {
              constexpr int kSteps = T2::kBox / 16;
#pragma unroll
              for (int jj = 0; jj < kSteps; ++jj) {
                const int kk = (blk - L::kNb1) * kSteps + jj;
                mma_bf16_ss(leader, d2, T2::desc_k(sb + L::oQ2 + T2::off_k(kk)), T2::desc_k(ks + jj * 32), idesc,
                            kk > 0);
              }
            }
            mma_commit(leader, bar_kempty(s));
          }
          if (!go) break;
          mma_commit(leader, bar_sfull(b));
        } else {
          const int s = j % L::kStages;
          const uint32_t ph = (j / L::kStages) & 1;
          if (!mbar_wait_warp(bar_kfull(s), ph, ctl)) break;
          if (!mbar_wait_warp(bar_sempty(b), bph ^ 1, ctl)) break;
          tc_fence_after();
          const uint32_t k1s = sb + L::oK + s * L::kStage, k2s = k1s + L::kK1;
#pragma unroll
          for (int kk = 0; kk < D1 / 16; ++kk) {
            const uint32_t o = T1::off_k(kk);
            mma_bf16_ss(leader, d1, T1::desc_k(sb + L::oQ1 + o), T1::desc_k(k1s + o), idesc, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D2 / 16; ++kk) {
            const uint32_t o = T2::off_k(kk);
            mma_bf16_ss(leader, d2, T2::desc_k(sb + L::oQ2 + o), T2::desc_k(k2s + o), idesc, kk > 0);
          }
          mma_commit(leader, bar_kempty(s));
          mma_commit(leader, bar_sfull(b));
        }
      }
    }
    // every MMA this warp issued has finished before TMEM is released
    mma_commit(leader, bar_done);
    mbar_drain(bar_done, 0, 1000000000ull);
  } else {
    // ---------------------------------------------------------------- statistics
    const int wg = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const int grow = q0 + row;
    const float c1 = a.scale1 * kLog2e, c2 = a.scale2 * kLog2e, nrho = -a.scale2 / a.scale1;
    const int lim = a.causal ? min(grow + off, a.NK - 1) : a.NK - 1;  // last visible key
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint64_t C1 = f2(c1, c1), C2 = f2(c2, c2), NR = f2(nrho, nrho);
    RowStats st{kNegBig, kNegBig, 0.f, 0.f, 0.f};
    const int col = wg * L::kCols;
    if constexpr (L::kCols == 32) {
      for (int j = 0; j < nkt; ++j) {
        const int b = j & 1;
        const uint32_t bph = (j >> 1) & 1;
        if (!mbar_wait_warp(bar_sfull(b), bph, ctl)) break;
        tc_fence_after();
        // this warpgroup's 32 columns of S1 and S2, summed against the
        // running maxima; a row whose sums reach 2^64 (rare after its first
        // tile) reads its columns again and folds them exactly.  S is
        // released after the fold: the other buffer keeps the MMA a tile ahead
        uint32_t x1[32], x2[32];
        const uint32_t t = tmem + lane_off + uint32_t(b * 256 + col);
        tmem_ld2x32(t, t + 128, x1, x2);
        const int k0 = (kt_lo + j) * kTile;
        const bool need_mask = (k0 + kTile > a.NK) || (a.causal && k0 + kTile - 1 > q0 + off);
        const int lr = need_mask ? lim - (k0 + col) : 0;
        if (j == 0) {  // no reference yet: every row folds its first tile exactly
          if (need_mask) fold_one<true>(st, x1, x2, C1, C2, NR, c1, c2, lr);
          else fold_one<false>(st, x1, x2, C1, C2, NR, c1, c2, 0);
        } else {
          const float nb1 = -st.m1 * c1, nb2 = -st.m2 * c2;
          float l1, l2, acc;
          if (need_mask) chunk_sums<true>(x1, x2, C1, C2, NR, f2(nb1, nb1), f2(nb2, nb2), lr, l1, l2, acc);
          else chunk_sums<false>(x1, x2, C1, C2, NR, f2(nb1, nb1), f2(nb2, nb2), 0, l1, l2, acc);
          const bool fast = l1 < 18446744073709551616.f && l2 < 18446744073709551616.f;  // 2^64
          if (fast) {
            st.l1 += l1;
            st.acc += acc;
            st.l2 += l2;
          }
          if (__any_sync(0xffffffffu, !fast)) {  // the TMEM loads are warp-wide
            tmem_ld2x32(t, t + 128, x1, x2);
            if (!fast) {
              if (need_mask) fold_one<true>(st, x1, x2, C1, C2, NR, c1, c2, lr);
              else fold_one<false>(st, x1, x2, C1, C2, NR, c1, c2, 0);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sempty(b));
      }
    } else {
      static_assert(L::kCols == 64, "fold_pair takes 64 columns");
      for (int j = 0; j < nkt; ++j) {
        const int b = j & 1;
        const uint32_t bph = (j >> 1) & 1;
        if (!mbar_wait_warp(bar_sfull(b), bph, ctl)) break;
        tc_fence_after();
        const int k0 = (kt_lo + j) * kTile;
        const bool need_mask = (k0 + kTile > a.NK) || (a.causal && k0 + kTile - 1 > q0 + off);
        // this warpgroup's 64 columns of S1 and S2 in one go, folded against
        // the running maxima; a row that finds a new maximum (rare after its
        // first tile) reads its columns again and folds them exactly.  S is
        // released after the fold: the other buffer keeps the MMA a tile ahead
        uint32_t xa1[32], xa2[32], xb1[32], xb2[32];
        const uint32_t t = tmem + lane_off + uint32_t(b * 256 + col);
        tmem_ld4x32(t, t + 128, t + 32, t + 160, xa1, xa2, xb1, xb2);
        const int lr = need_mask ? lim - (k0 + col) : 0;
        // no reference yet on the first tile: every row folds it exactly
        const bool fast =
            j > 0 && (need_mask ? fold_pair_fast<true>(st, xa1, xa2, xb1, xb2, C1, C2, NR, c1, c2, lr)
                                : fold_pair_fast<false>(st, xa1, xa2, xb1, xb2, C1, C2, NR, c1, c2, 0));
        if (j == 0) {
          if (need_mask) fold_pair<true>(st, xa1, xa2, xb1, xb2, C1, C2, NR, c1, c2, lr);
          else fold_pair<false>(st, xa1, xa2, xb1, xb2, C1, C2, NR, c1, c2, 0);
        } else if (__any_sync(0xffffffffu, !fast)) {  // the TMEM loads are warp-wide
          tmem_ld4x32(t, t + 128, t + 32, t + 160, xa1, xa2, xb1, xb2);
          if (!fast) {
            if (need_mask) fold_pair<true>(st, xa1, xa2, xb1, xb2, C1, C2, NR, c1, c2, lr);
            else fold_pair<false>(st, xa1, xa2, xb1, xb2, C1, C2, NR, c1, c2, 0);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sempty(b));
      }
    }
    // merge the column shares of every row (warpgroups 1.. -> warpgroup 0)
    // with the same algebra as the key-split reduce
    float* mg = reinterpret_cast<float*>(smem + L::oMerge);
    if (wg > 0) {
      float* o = mg + (wg - 1) * kTile * 5 + row * 5;
      o[0] = st.m1;
      o[1] = st.l1;
      o[2] = st.acc;
      o[3] = st.m2;
      o[4] = st.l2;
    }
    named_bar_sync(1, 32 * L::kStatWarps);
    if (wg == 0 && !*abort_flag && grow < a.NQ) {
      float M1 = st.m1, M2 = st.m2;
#pragma unroll
      for (int w = 0; w < L::kWGs - 1; ++w) {
        M1 = fmaxf(M1, mg[w * kTile * 5 + row * 5 + 0]);
        M2 = fmaxf(M2, mg[w * kTile * 5 + row * 5 + 3]);
      }
      const float e1 = ex2((st.m1 - M1) * c1), e2 = ex2((st.m2 - M2) * c2);
      float L1 = st.l1 * e1, A = st.acc * e1, L2 = st.l2 * e2;
#pragma unroll
      for (int w = 0; w < L::kWGs - 1; ++w) {
        const float* o = mg + w * kTile * 5 + row * 5;
        const float g1 = ex2((o[0] - M1) * c1), g2 = ex2((o[3] - M2) * c2);
        L1 = fmaf(o[1], g1, L1);
        A = fmaf(o[2], g1, A);
        L2 = fmaf(o[4], g2, L2);
      }
      const size_t rows = size_t(a.BH) * a.NQ;
      const size_t idx = size_t(bh) * a.NQ + grow;
      if (!SKL_CHECK(a.status, idx < rows && split < a.num_splits)) {
        // (debug build) out-of-range row or split: nothing is written
      } else if (a.partial != nullptr) {
        float* p = a.partial + size_t(split) * 5 * rows + idx;
        p[0 * rows] = a.scale1 * M1;
        p[1 * rows] = L1;
        p[2 * rows] = a.scale1 * A;
        p[3 * rows] = a.scale2 * M2;
        p[4 * rows] = L2;
      } else {
        const float lse1 = a.scale1 * M1 + logf(L1);
        const float lse2 = a.scale2 * M2 + logf(L2);
        a.lse1[idx] = lse1;
        a.lse2[idx] = lse2;
        a.kl[idx] = a.scale1 * A / L1 + lse2 - lse1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


template <int D1, int D2>
inline int launch_fwd_t(const TMaps& m, const FwdArgs& a, cudaStream_t st) {
  using L = FwdLayout<D1, D2>;
  auto kern = fwd_kernel<D1, D2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int nqt = (a.NQ + kTile - 1) / kTile;
  dim3 grid(nqt, a.BH, a.num_splits);
  kern<<<grid, L::kThreads, L::kAlloc, st>>>(m.q1, m.k1, m.q2, m.k2, a);
  return cudaGetLastError();
}


}  // namespace skl
