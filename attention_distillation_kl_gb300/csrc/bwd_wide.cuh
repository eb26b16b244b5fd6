// Backward for head dims above 128 (tile width 192 or 256 on either side).
//
// The fused backward keeps S1, S2, dK and dQ in TMEM (256 + 2 dg columns) and
// both sides' K tiles plus two Q tiles in shared memory; above 128 neither
// fits.  This path takes the deterministic structure instead: two passes
// that each hold one gradient accumulator, recompute S1 and S2 (StreamKL
// article, "Backward": P rebuilt from the saved LSEs) and stream the
// operands they visit through a ring of 64-column blocks:
//
//   pass 0 (dK): one CTA per 128-key tile.  Owner operands K1, K2 of the
//                tile stay in shared memory; for every query tile that sees
//                it the blocks of Q1, Q2 (for S) and of Q_g (for
//                dK[:, c] += dS^T Q_g[:, c], one 64-column chunk c per block)
//                stream through the ring.  dK is stored once at the end
//                (grouped key heads: ordered launches, the first stores and
//                the others add).
//   pass 1 (dQ): one CTA per 128-query tile (longest rows first).  Owner
//                operands Q1, Q2; for every visible key tile the blocks of
//                K1, K2 and K_g stream (dQ[:, c] += dS K_g[:, c]).  dQ is
//                stored once.
//
// No atomics anywhere, so results are bitwise reproducible.  TMEM: S1 [0,128),
// S2 [128,256), the accumulator [256, 256 + DG).  Warps 0-7 form dS (thread =
// query row, as in the fused kernel) and at the end store the accumulator;
// warp 8 issues the TMA loads; warp 9 owns TMEM and runs the MMA loop (one
// elected lane issues).  The 512 TMEM columns hold one S pair, so the dS
// warps take their whole share of S into registers and release it at once:
// the S products of tile v then run while dS of tile v - 1 is formed, and
// the gradient product of tile v - 1 follows them (the ring carries the
// blocks in that order).
#pragma once

#include "bwd_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace skl {

constexpr int kWideThreads = 320;

template <int D1, int D2, int MODE>
struct WideLayout {
  static constexpr int DG = MODE == STREAMKL_GRAD_P2 ? D2 : D1;
  static constexpr uint32_t kO1 = kTile * D1 * 2, kO2 = kTile * D2 * 2;  // owner tiles of sides 1, 2
  static constexpr uint32_t kDS = kTile * kTile * 2;
  static constexpr uint32_t kSlot = 16384;  // one operand block (at most 128 rows x 64 bf16)
  static constexpr uint32_t oO1 = 0, oO2 = kO1, oDS = kO1 + kO2, oRing = oDS + kDS;
  static constexpr int kSlotsFit = int((230400u - oRing) / kSlot);
  static constexpr int kSlots = kSlotsFit > 8 ? 8 : kSlotsFit;
  static constexpr int kNb1 = OpTile<D1>::kBlocks, kNb2 = OpTile<D2>::kBlocks, kNbg = OpTile<DG>::kBlocks;
  static constexpr int kPerVisit = kNb1 + kNb2 + kNbg;  // ring blocks per visited tile
  static constexpr uint32_t oBar = oRing + kSlots * kSlot;
  enum { B_OFULL = 0, B_VFULL = 1, B_VEMPTY = 9, B_SFULL = 17, B_SFREE, B_DSFULL, B_DSEMPTY, B_GFULL, B_DONE,
         kNumBars };
  static constexpr uint32_t oMisc = oBar + kNumBars * 8;
  static constexpr uint32_t kBytes = oMisc + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static_assert(kSlots >= 2, "the block ring needs two slots");
  static_assert(kSlots <= 8, "barrier table holds eight slots");
  static_assert(kAlloc <= 232448, "over the 227 KB shared memory limit");
};

template <int D1, int D2, int MODE, int PASS>
__global__ void __launch_bounds__(kWideThreads, 1)
    bwd_wide_kernel(const __grid_constant__ CUtensorMap tq1, const __grid_constant__ CUtensorMap tk1,
                    const __grid_constant__ CUtensorMap tq2, const __grid_constant__ CUtensorMap tk2,
                    const BwdArgs a) {
  using L = WideLayout<D1, D2, MODE>;
  constexpr int DG = L::DG;
  constexpr bool kP2 = MODE == STREAMKL_GRAD_P2;
  constexpr bool kDK = PASS == 0;
  using T1 = OpTile<D1>;
  using T2 = OpTile<D2>;
  using TG = OpTile<DG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int gg = kP2 ? a.g2 : a.g1;  // query heads per gradient-side key head
  const int off = a.NK - a.NQ;
  const int nqt = (a.NQ + kTile - 1) / kTile;
  // pass 0: key tile kt, visitors = query tiles qt_lo .. nqt - 1
  // pass 1: query tile qt (longest rows first), visitors = key tiles 0 .. nv - 1
  // the launch's heads in groups whose tiles interleave, longest first
  int hy, tx;
  grouped_unit(int(blockIdx.y) * int(gridDim.x) + int(blockIdx.x), int(gridDim.y), int(gridDim.x), a.head_group,
               hy, tx);
  int bh, k0 = 0, q0 = 0, qt_lo = 0, nv;
  if constexpr (kDK) {
    bh = a.hsel < 0 ? hy : hy * gg + a.hsel;
    k0 = tx * kTile;
    qt_lo = a.causal ? max(0, k0 - off) / kTile : 0;
    nv = nqt - qt_lo;
  } else {
    bh = hy;
    const int qt = a.causal ? (nqt - 1 - tx) : tx;
    q0 = qt * kTile;
    const int kend = a.causal ? min(q0 + kTile, a.NQ) + off : a.NK;
    nv = (kend + kTile - 1) / kTile;
  }

  auto bar = [&](int id) { return sb + L::oBar + 8u * id; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oMisc + 4);
  const Ctl ctl{abort_flag, a.status};

  if (threadIdx.x == 0) {
    for (int b = 0; b < L::kNumBars; ++b) mbar_init(bar(b), (b == L::B_DSFULL || b == L::B_SFREE) ? 8u : 1u);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s1 = tmem, t_s2 = tmem + 128, t_g = tmem + 256;

  if (warp == 8) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && nv > 0) {
      tma_prefetch_desc(&tq1);
      tma_prefetch_desc(&tk1);
      tma_prefetch_desc(&tq2);
      tma_prefetch_desc(&tk2);
      mbar_arrive_expect_tx(bar(L::B_OFULL), L::kO1 + L::kO2);
      if constexpr (kDK) {
        T1::load(sb + L::oO1, &tk1, bar(L::B_OFULL), k0, bh / a.g1);
        T2::load(sb + L::oO2, &tk2, bar(L::B_OFULL), k0, bh / a.g2);
      } else {
        T1::load(sb + L::oO1, &tq1, bar(L::B_OFULL), q0, bh);
        T2::load(sb + L::oO2, &tq2, bar(L::B_OFULL), q0, bh);
      }
      // visitor blocks in the order the MMA loop takes them: side 1, side 2
      // (for S), then the gradient side again (for the gradient product)
      const CUtensorMap* m1 = kDK ? &tq1 : &tk1;
      const CUtensorMap* m2 = kDK ? &tq2 : &tk2;
      const CUtensorMap* mg = kP2 ? m2 : m1;
      const int z1 = kDK ? bh : bh / a.g1, z2 = kDK ? bh : bh / a.g2, zg = kP2 ? z2 : z1;
      int issued = 0;
      bool go = true;
      // one visited tile's blocks: its S operands (side 1, side 2) or its
      // gradient operand, into the ring in the order the MMA loop takes them
      auto put_blocks = [&](int v, bool grad) {
        const int r0 = kDK ? (qt_lo + v) * kTile : v * kTile;  // first row of the visited tile
        const int b0 = grad ? L::kNb1 + L::kNb2 : 0, b1 = grad ? L::kPerVisit : L::kNb1 + L::kNb2;
#pragma unroll 1
        for (int blk = b0; blk < b1 && go; ++blk) {
          const int u = issued, s = u % L::kSlots;
          if (!mbar_wait_polled(bar(L::B_VEMPTY + s), ((u / L::kSlots) & 1) ^ 1, ctl)) {
            go = false;
            break;
          }
          const uint32_t dst = sb + L::oRing + s * L::kSlot;
          if (!SKL_CHECK(a.status, dst + L::kSlot <= sb + L::oBar && r0 < (kDK ? a.NQ : a.NK) + kTile)) {
            go = false;
            break;
          }
          if (blk < L::kNb1) {
            mbar_arrive_expect_tx(bar(L::B_VFULL + s), T1::kBlockBytes);
            tma_load_3d(dst, m1, bar(L::B_VFULL + s), blk * T1::kBox, r0, z1);
          } else if (blk < L::kNb1 + L::kNb2) {
            mbar_arrive_expect_tx(bar(L::B_VFULL + s), T2::kBlockBytes);
            tma_load_3d(dst, m2, bar(L::B_VFULL + s), (blk - L::kNb1) * T2::kBox, r0, z2);
          } else {
            mbar_arrive_expect_tx(bar(L::B_VFULL + s), TG::kBlockBytes);
            tma_load_3d(dst, mg, bar(L::B_VFULL + s), (blk - L::kNb1 - L::kNb2) * TG::kBox, r0, zg);
          }
          issued = u + 1;
        }
      };
      // the S products of tile v go before the gradient product of tile v - 1
      for (int v = 0; v < nv && go; ++v) {
        put_blocks(v, false);
        if (v > 0) put_blocks(v - 1, true);
      }
      if (go) put_blocks(nv - 1, true);
      if (*abort_flag) {  // let the copies already started land before the CTA exits
        const uint64_t lim = 200000000ull;
        mbar_drain(bar(L::B_OFULL), 0, lim);
        for (int u = issued > L::kSlots ? issued - L::kSlots : 0; u < issued; ++u)
          mbar_drain(bar(L::B_VFULL + u % L::kSlots), (u / L::kSlots) & 1, lim);
      }
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    // (the whole warp runs the loop; the elected lane issues)
    const uint32_t leader = elect_one();
    constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);
    // gradient product per 64-column (or 32-column) chunk of the head dim:
    // pass 0 A = dS^T (M-major), pass 1 A = dS (K-major); B = the visitor block, N-major
    constexpr uint32_t id_g = idesc_bf16(128, TG::kBox, kDK ? 1 : 0, 1);
    const uint64_t dsm = sdesc_sw128(sb + L::oDS, kTile * 128, 1024);  // dS^T, M-major
    const uint64_t dsk = sdesc_sw128(sb + L::oDS, 16, 1024);           // dS, K-major
    bool done = false;
    int u = 0;  // ring blocks taken, in the producer's order
    // S1, S2 of visited tile v into TMEM (the dS warps have read the previous S)
    auto s_products = [&](int v) {
      (void)v;
#pragma unroll 1
      for (int blk = 0; blk < L::kNb1 + L::kNb2; ++blk, ++u) {
        const int s = u % L::kSlots;
        if (!mbar_wait_warp(bar(L::B_VFULL + s), (u / L::kSlots) & 1, ctl)) return false;
        tc_fence_after();
        const uint32_t vs = sb + L::oRing + s * L::kSlot;  // visitor block
        // owner operand block kk / steps at offset off_k(kk); visitor block step jj at jj * 32
        auto s_steps = [&](auto tile, uint32_t d, uint32_t owner, int b) {
          using T = decltype(tile);
          constexpr int kSteps = T::kBox / 16;
#pragma unroll
          for (int jj = 0; jj < kSteps; ++jj) {
            const int kk = b * kSteps + jj;
            const uint64_t od = T::desc_k(owner + T::off_k(kk)), vd = T::desc_k(vs + jj * 32);
            // S = Q K^T with queries as M: pass 0 visits Q (A), pass 1 visits K (B)
            if constexpr (kDK) mma_bf16_ss(leader, d, vd, od, id_s, kk > 0);
            else mma_bf16_ss(leader, d, od, vd, id_s, kk > 0);
          }
        };
        if (blk < L::kNb1) s_steps(T1{}, t_s1, sb + L::oO1, blk);
        else s_steps(T2{}, t_s2, sb + L::oO2, blk - L::kNb1);
        mma_commit(leader, bar(L::B_VEMPTY + s));
      }
      mma_commit(leader, bar(L::B_SFULL));
      return true;
    };
    // the gradient product of visited tile v, once its dS is in shared memory;
    // the dS tile is free again when these products are done
    auto grad_product = [&](int v) {
      if (!mbar_wait_warp(bar(L::B_DSFULL), v & 1, ctl)) return false;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < L::kNbg; ++c, ++u) {
        const int s = u % L::kSlots;
        if (!mbar_wait_warp(bar(L::B_VFULL + s), (u / L::kSlots) & 1, ctl)) return false;
        tc_fence_after();
        const uint64_t gd = TG::desc_n(sb + L::oRing + s * L::kSlot);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t ad = kDK ? sdesc_add(dsm, kk * 2048)
                                  : sdesc_add(dsk, (kk >> 2) * (kTile * 128) + (kk & 3) * 32);
          mma_bf16_ss(leader, t_g + c * TG::kBox, ad, sdesc_add(gd, TG::off_n(kk)), id_g,
                      (v > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(leader, bar(L::B_VEMPTY + s));
      }
      mma_commit(leader, bar(L::B_DSEMPTY));
      return true;
    };
    if (nv > 0 && mbar_wait_warp(bar(L::B_OFULL), 0, ctl) && s_products(0)) {
      bool go = true;
      for (int v = 1; v < nv && go; ++v) {
        // S of tile v as soon as the dS warps hold S of tile v - 1 in
        // registers, so it runs while they form dS of tile v - 1
        go = mbar_wait_warp(bar(L::B_SFREE), (v - 1) & 1, ctl) && s_products(v) && grad_product(v - 1);
      }
      done = go && grad_product(nv - 1) && !*abort_flag;
    }
    if (done) mma_commit(leader, bar(L::B_GFULL));
    // every MMA this warp issued has finished before TMEM is released
    mma_commit(leader, bar(L::B_DONE));
    mbar_drain(bar(L::B_DONE), 0, 1000000000ull);
  } else {
    // ---------------------------------------------------------------- dS, then the accumulator
    const int wg = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float c1 = a.scale1 * kLog2e, c2 = a.scale2 * kLog2e, nr = -a.scale2 / a.scale1;
    const uint64_t C1 = f2(c1, c1), C2 = f2(c2, c2), S1 = f2(a.scale1, a.scale1), NR = f2(nr, nr);
    const float sg = kP2 ? a.scale2 : a.scale1;  // softmax scale of the gradient side
    // per-row parameters of query row qi (see ds_chunk_row)
    auto params = [&](int qi, float& na, float& nb, float& ws) {
      na = -INFINITY;
      nb = kP2 ? -INFINITY : 0.f;
      ws = 0.f;
      if (qi < a.NQ) {
        const size_t idx = size_t(bh) * a.NQ + qi;
        const float l1 = a.lse1[idx];
        na = -l1 * kLog2e;
        ws = sg * a.dkl[idx];
        nb = kP2 ? -a.lse2[idx] * kLog2e : -(l1 - a.lse2[idx] + a.kl[idx]);
      }
    };
    float na, nb, ws;
    params(kDK ? qt_lo * kTile + row : q0 + row, na, nb, ws);
    int v = 0;
    for (; v < nv; ++v) {
      const int tq0 = kDK ? (qt_lo + v) * kTile : q0;  // query tile of this step
      const int tk0 = kDK ? k0 : v * kTile;            // key tile of this step
      const uint64_t NA = f2(na, na), NB = f2(nb, nb), WW = f2(ws, ws);
      if (kDK && v + 1 < nv) params(tq0 + kTile + row, na, nb, ws);  // the next tile's rows
      if (!mbar_wait_warp(bar(L::B_SFULL), v & 1, ctl)) break;
      tc_fence_after();
      const int lim = (a.causal ? min(tq0 + row + off, a.NK - 1) : a.NK - 1) - tk0;  // last visible key
      const bool need_mask = (tk0 + kTile > a.NK) || (a.causal && tq0 < tk0 + kTile - 1 - off);
      // this warp's 64 columns of S1 and S2 into registers, then S is free
      // for the next tile's products while dS is formed
      const int col = wg * 64;
      uint32_t x1a[32], x2a[32], x1b[32], x2b[32];
      tmem_ld2x32(t_s1 + lane_off + col, t_s2 + lane_off + col, x1a, x2a);
      tmem_ld2x32(t_s1 + lane_off + col + 32, t_s2 + lane_off + col + 32, x1b, x2b);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_SFREE));
      uint32_t dsr[32];
      if (need_mask) {
        ds_chunk_row<MODE, true>(x1a, x2a, C1, C2, S1, NR, NA, NB, WW, lim - col, dsr);
        ds_chunk_row<MODE, true>(x1b, x2b, C1, C2, S1, NR, NA, NB, WW, lim - col - 32, dsr + 16);
      } else {
        ds_chunk_row<MODE, false>(x1a, x2a, C1, C2, S1, NR, NA, NB, WW, 0, dsr);
        ds_chunk_row<MODE, false>(x1b, x2b, C1, C2, S1, NR, NA, NB, WW, 0, dsr + 16);
      }
      // the previous tile's gradient product is done reading the dS tile
      if (v > 0 && !mbar_wait_warp(bar(L::B_DSEMPTY), (v - 1) & 1, ctl)) break;
      store_half_row_sw128(sb + L::oDS, row, wg, dsr);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_DSFULL));
    }
    // the accumulator: rows are keys (pass 0) or queries (pass 1); warpgroup
    // wg stores the 32-column chunks ch = wg, wg + 2, ...
    if constexpr (kDK) {
      const int dk_how = (gg == 1 || a.hsel <= 0) ? kDkStore : kDkAdd;
      const int kj = k0 + row;
      float* dst = a.dk + (size_t(bh / gg) * a.NK + kj) * a.dg;
      if (nv > 0 && v == nv && mbar_wait_warp(bar(L::B_GFULL), 0, ctl)) {
        tc_fence_after();
        for (int ch = wg; ch < DG / 32; ch += 2) {
          uint32_t x[32];
          tmem_ld32(t_g + lane_off + ch * 32, x);
          if (kj < a.NK && SKL_CHECK(a.status, bh / gg < a.BH / gg && a.dg <= DG)) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              if (ch * 32 + e < a.dg)
                put_dk4(dst + ch * 32 + e,
                        make_float4(__uint_as_float(x[e]), __uint_as_float(x[e + 1]), __uint_as_float(x[e + 2]),
                                    __uint_as_float(x[e + 3])),
                        dk_how);
          }
        }
      } else if (nv == 0 && dk_how == kDkStore && kj < a.NK) {
        // no query row sees this key tile: its dK is zero
        for (int e = wg * 4; e < a.dg; e += 8)
          *reinterpret_cast<float4*>(dst + e) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
      const int qi = q0 + row;
      float* dst = a.dq + (size_t(bh) * a.NQ + qi) * a.dg;
      if (nv > 0 && v == nv && mbar_wait_warp(bar(L::B_GFULL), 0, ctl)) {
        tc_fence_after();
        for (int ch = wg; ch < DG / 32; ch += 2) {
          uint32_t x[32];
          tmem_ld32(t_g + lane_off + ch * 32, x);
          if (qi < a.NQ && SKL_CHECK(a.status, bh < a.BH && a.dg <= DG)) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              if (ch * 32 + e < a.dg)
                *reinterpret_cast<float4*>(dst + ch * 32 + e) =
                    make_float4(__uint_as_float(x[e]), __uint_as_float(x[e + 1]), __uint_as_float(x[e + 2]),
                                __uint_as_float(x[e + 3]));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D1, int D2, int MODE, int PASS>
inline int launch_wide_t(const TMaps& m, const BwdArgs& a, cudaStream_t st) {
  using L = WideLayout<D1, D2, MODE>;
  auto kern = bwd_wide_kernel<D1, D2, MODE, PASS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int gg = MODE == STREAMKL_GRAD_P2 ? a.g2 : a.g1;
  dim3 grid;
  if (PASS == 0) grid = dim3((a.NK + kTile - 1) / kTile, a.hsel < 0 ? a.BH : a.BH / gg);
  else grid = dim3((a.NQ + kTile - 1) / kTile, a.BH);
  kern<<<grid, kWideThreads, L::kAlloc, st>>>(m.q1, m.k1, m.q2, m.k2, a);
  return cudaGetLastError();
}

}  // namespace skl
