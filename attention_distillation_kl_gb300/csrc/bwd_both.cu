// Both-sides backward: the gradient of L = sum_i dKL_i KL_i with respect to
// both distributions from one recompute of S1 and S2 (StreamKL article,
// "Backward": the two modes share the recomputed P1, P2; running both in one
// pass is a widening of the method, not a mode the pages name):
//   dS2 = dKL (P2 - P1)                 -> dQ2 = s2 dS2 K2, dK2 = s2 dS2^T Q2
//   dS1 = dKL P1 (r - KL), r from logits -> dQ1 = s1 dS1 K1, dK1 = s1 dS1^T Q1
// Built for tile widths D = 64 or 32 (d1 = d2 = a.dg <= D; columns past a.dg
// are zero-filled by the TMA and not written), where the four accumulators fit
// next to S1 and S2 in the 512 TMEM columns (each takes D columns of a
// 64-column slot):
//   S1 [0,128)  S2 [128,256)  dK1 256  dK2 320  dQ1 384  dQ2 448
// One CTA owns a 128-key tile and walks the query tiles that see it, like the
// single-side fused kernel.  16 warps:
//   warps 0-7   thread = query row: P1, P2 once, then dS1 and dS2 (bf16, two
//               swizzled tiles), warps 0-3 key columns 0-63, warps 4-7 64-127
//   warps 8-11  drain dQ1 and dQ2 (TMEM -> 2 KB swizzled boxes -> TMA bulk
//               reduce-add into each side's fp32 dQ); finally dK1 and dK2
//   warp 12     TMA: K1, K2 once; Q1 and Q2 of each query tile (double buffer)
//   warp 13     TMEM owner, S issuer
//   warp 14     dK issuer: dK1 += dS1^T Q1, dK2 += dS2^T Q2
//   warp 15     dQ issuer: dQ1 = dS1 K1, dQ2 = dS2 K2
#include "bwd_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace skl {

namespace {

constexpr int kBothThreads = 512;
constexpr int kBothBoxes = 4;  // dQ staging boxes per epilogue warp

template <int D_>
struct BothLayout {
  static constexpr int D = D_;
  static constexpr uint32_t kDS = kTile * kTile * 2;  // one bf16 dS tile
  static constexpr uint32_t kK = kTile * D * 2, kQ = kTile * D * 2;
  static constexpr uint32_t oDS1 = 0, oDS2 = kDS, oK1 = 2 * kDS, oK2 = oK1 + kK;
  static constexpr uint32_t oQ1 = oK2 + kK, oQ2 = oQ1 + 2 * kQ;  // two buffers each
  static constexpr uint32_t oStage = oQ2 + 2 * kQ;
  static constexpr uint32_t oBar = oStage + 4 * kBothBoxes * 2048;
  enum {
    B_KFULL, B_QFULL0, B_QFULL1, B_QEMPTY0, B_QEMPTY1, B_SFULL, B_SFREE, B_DSFULL, B_DSEMPTY, B_DQFULL,
    B_DQEMPTY, B_DKFULL, B_DONE, kNumBars
  };
  static constexpr uint32_t oMisc = oBar + kNumBars * 8;
  static constexpr uint32_t kBytes = oMisc + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "over the 227 KB shared memory limit");
};

template <int D_>
__global__ void __launch_bounds__(kBothThreads, 1)
    bwd_both_kernel(const __grid_constant__ CUtensorMap tq1, const __grid_constant__ CUtensorMap tk1,
                    const __grid_constant__ CUtensorMap tq2, const __grid_constant__ CUtensorMap tk2,
                    const __grid_constant__ CUtensorMap tdq1, const __grid_constant__ CUtensorMap tdq2,
                    const BwdArgs a) {
  using L = BothLayout<D_>;
  using T = OpTile<D_>;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int bh, kt;  // heads in groups whose key tiles interleave, longest sweeps first
  grouped_unit(int(blockIdx.y) * int(gridDim.x) + int(blockIdx.x), a.BH, int(gridDim.x), a.head_group, bh, kt);
  const int k0 = kt * kTile;
  const int off = a.NK - a.NQ;
  const int nqt = (a.NQ + kTile - 1) / kTile;
  const int qt_lo = a.causal ? max(0, k0 - off) / kTile : 0;  // first query tile that sees a key here
  const int n = nqt - qt_lo;

  auto bar = [&](int id) { return sb + L::oBar + 8u * id; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oMisc + 4);
  const Ctl ctl{abort_flag, a.status};

  if (threadIdx.x == 0) {
    for (int b = 0; b < L::kNumBars; ++b) {
      uint32_t count = 1;
      if (b == L::B_SFREE || b == L::B_DSFULL) count = 8;  // one per dS warp
      if (b == L::B_DQEMPTY) count = 4;                    // one per epilogue warp
      if (b == L::B_DSEMPTY) count = 2;                    // the dK and dQ issuers
      if (b == L::B_DONE) count = 3;                       // one per MMA issuer
      mbar_init(bar(b), count);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s1 = tmem, t_s2 = tmem + 128, t_dk1 = tmem + 256, t_dk2 = tmem + 320;
  const uint32_t t_dq = tmem + 384;  // dQ1 [384, 448), dQ2 [448, 512)

  if (warp == 12) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tq1);
      tma_prefetch_desc(&tk1);
      tma_prefetch_desc(&tq2);
      tma_prefetch_desc(&tk2);
      mbar_arrive_expect_tx(bar(L::B_KFULL), 2 * L::kK);
      T::load(sb + L::oK1, &tk1, bar(L::B_KFULL), k0, bh);
      T::load(sb + L::oK2, &tk2, bar(L::B_KFULL), k0, bh);
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int g = i & 1;
        if (!mbar_wait_polled(bar(L::B_QEMPTY0 + g), ((i >> 1) & 1) ^ 1, ctl)) break;
        mbar_arrive_expect_tx(bar(L::B_QFULL0 + g), 2 * L::kQ);
        const int q0 = (qt_lo + i) * kTile;
        T::load(sb + L::oQ1 + g * L::kQ, &tq1, bar(L::B_QFULL0 + g), q0, bh);
        T::load(sb + L::oQ2 + g * L::kQ, &tq2, bar(L::B_QFULL0 + g), q0, bh);
        issued = i + 1;
      }
      if (*abort_flag) {  // let the copies already started land before the CTA exits
        const uint64_t lim = 200000000ull;
        mbar_drain(bar(L::B_KFULL), 0, lim);
        for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
          mbar_drain(bar(L::B_QFULL0 + (i & 1)), (i >> 1) & 1, lim);
      }
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------------- S issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);
      const uint64_t k1d = T::desc_k(sb + L::oK1), k2d = T::desc_k(sb + L::oK2);
      bool ok = n > 0 && mbar_wait_polled(bar(L::B_KFULL), 0, ctl);
      for (int i = 0; ok && i < n; ++i) {
        const int g = i & 1;
        if (!mbar_wait_polled(bar(L::B_SFREE), (i & 1) ^ 1, ctl)) break;
        if (!mbar_wait_polled(bar(L::B_QFULL0 + g), (i >> 1) & 1, ctl)) break;
        tc_fence_after();
        const uint64_t q1d = T::desc_k(sb + L::oQ1 + g * L::kQ);
        const uint64_t q2d = T::desc_k(sb + L::oQ2 + g * L::kQ);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(1u, t_s1, sdesc_add(q1d, T::off_k(kk)), sdesc_add(k1d, T::off_k(kk)), id_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(1u, t_s2, sdesc_add(q2d, T::off_k(kk)), sdesc_add(k2d, T::off_k(kk)), id_s, kk > 0);
        mma_commit(1u, bar(L::B_SFULL));
      }
      // every MMA of every issuer has finished before TMEM is released
      mma_commit(1u, bar(L::B_DONE));
      mbar_drain(bar(L::B_DONE), 0, 1000000000ull);
    }
  } else if (warp == 14) {
    // ---------------------------------------------------------------- dK issuer
    if (lane == 0) {
      constexpr uint32_t id_dk = idesc_bf16(128, D, 1, 1);  // A = dS^T M-major, B = Q N-major
      const uint64_t ds1 = sdesc_sw128(sb + L::oDS1, kTile * 128, 1024);
      const uint64_t ds2 = sdesc_sw128(sb + L::oDS2, kTile * 128, 1024);
      int t = 0;
      if (n > 0 && mbar_wait_polled(bar(L::B_KFULL), 0, ctl)) {
        for (; t < n; ++t) {
          if (!mbar_wait_polled(bar(L::B_DSFULL), t & 1, ctl)) break;
          tc_fence_after();
          const int g = t & 1;
          const uint64_t q1n = T::desc_n(sb + L::oQ1 + g * L::kQ);
          const uint64_t q2n = T::desc_n(sb + L::oQ2 + g * L::kQ);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss(1u, t_dk1, sdesc_add(ds1, kk * 2048), sdesc_add(q1n, T::off_n(kk)), id_dk,
                        (t > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss(1u, t_dk2, sdesc_add(ds2, kk * 2048), sdesc_add(q2n, T::off_n(kk)), id_dk,
                        (t > 0 || kk > 0) ? 1u : 0u);
          mma_commit(1u, bar(L::B_QEMPTY0 + g));  // S and dK are done with Q1, Q2 of tile t
          mma_commit(1u, bar(L::B_DSEMPTY));
        }
      }
      if (n > 0 && t == n && !*abort_flag) mma_commit(1u, bar(L::B_DKFULL));
      mma_commit(1u, bar(L::B_DONE));  // the TMEM owner drains it before releasing TMEM
    }
  } else if (warp == 15) {
    // ---------------------------------------------------------------- dQ issuer
    if (lane == 0) {
      constexpr uint32_t id_dq = idesc_bf16(128, D, 0, 1);  // A = dS K-major, B = K N-major
      const uint64_t ds1 = sdesc_sw128(sb + L::oDS1, 16, 1024), ds2 = sdesc_sw128(sb + L::oDS2, 16, 1024);
      const uint64_t k1n = T::desc_n(sb + L::oK1);
      const uint64_t k2n = T::desc_n(sb + L::oK2);
      if (n > 0 && mbar_wait_polled(bar(L::B_KFULL), 0, ctl)) {
        for (int t = 0; t < n; ++t) {
          if (!mbar_wait_polled(bar(L::B_DSFULL), t & 1, ctl)) break;
          if (!mbar_wait_polled(bar(L::B_DQEMPTY), (t & 1) ^ 1, ctl)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t ao = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
            mma_bf16_ss(1u, t_dq, sdesc_add(ds1, ao), sdesc_add(k1n, T::off_n(kk)), id_dq, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t ao = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
            mma_bf16_ss(1u, t_dq + 64, sdesc_add(ds2, ao), sdesc_add(k2n, T::off_n(kk)), id_dq, kk > 0 ? 1u : 0u);
          }
          mma_commit(1u, bar(L::B_DSEMPTY));
          mma_commit(1u, bar(L::B_DQFULL));
        }
      }
      mma_commit(1u, bar(L::B_DONE));  // the TMEM owner drains it before releasing TMEM
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------- dS1, dS2 (thread = query row)
    const int wg = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float c1 = a.scale1 * kLog2e, c2 = a.scale2 * kLog2e, nr = -a.scale2 / a.scale1;
    const uint64_t C1 = f2(c1, c1), C2 = f2(c2, c2), S1 = f2(a.scale1, a.scale1), NR = f2(nr, nr);
    // per-row parameters of query tile i (see ds_chunk_row_both), loaded a tile ahead
    auto params = [&](int i, float& na, float& nb2, float& nb1, float& w) {
      const int qi = (qt_lo + i) * kTile + row;
      na = -INFINITY;
      nb2 = -INFINITY;
      nb1 = 0.f;
      w = 0.f;
      if (qi < a.NQ) {
        const size_t idx = size_t(bh) * a.NQ + qi;
        const float l1 = a.lse1[idx], l2 = a.lse2[idx];
        na = -l1 * kLog2e;
        nb2 = -l2 * kLog2e;
        nb1 = -(l1 - l2 + a.kl[idx]);
        w = a.dkl[idx];
      }
    };
    float na, nb2, nb1, w;
    if (n > 0) params(0, na, nb2, nb1, w);
    for (int i = 0; i < n; ++i) {
      const int q0 = (qt_lo + i) * kTile;
      const uint64_t NA = f2(na, na), NB2 = f2(nb2, nb2), NB1 = f2(nb1, nb1);
      const uint64_t W2 = f2(a.scale2 * w, a.scale2 * w), W1 = f2(a.scale1 * w, a.scale1 * w);
      if (i + 1 < n) params(i + 1, na, nb2, nb1, w);
      if (!mbar_wait_warp(bar(L::B_SFULL), i & 1, ctl)) break;
      tc_fence_after();
      const int lim = (a.causal ? min(q0 + row + off, a.NK - 1) : a.NK - 1) - k0;  // last visible key
      const bool need_mask = (k0 + kTile > a.NK) || (a.causal && q0 < k0 + kTile - 1 - off);
      bool ok = true;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int col = wg * 64 + ch * 32;
        uint32_t x1[32], x2[32], d1r[16], d2r[16];
        tmem_ld2x32(t_s1 + lane_off + col, t_s2 + lane_off + col, x1, x2);
        if (ch == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::B_SFREE));
        }
        if (need_mask)
          ds_chunk_row_both<true>(x1, x2, C1, C2, S1, NR, NA, NB2, NB1, W2, W1, lim - col, d1r, d2r);
        else
          ds_chunk_row_both<false>(x1, x2, C1, C2, S1, NR, NA, NB2, NB1, W2, W1, 0, d1r, d2r);
        // the previous tile's products must be done reading dS before it is replaced
        if (ch == 0 && !mbar_wait_warp(bar(L::B_DSEMPTY), (i & 1) ^ 1, ctl)) {
          ok = false;
          break;
        }
        store_cols32_sw128(sb + L::oDS1, row, col, d1r);
        store_cols32_sw128(sb + L::oDS2, row, col, d2r);
      }
      if (!ok) break;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_DSFULL));
    }
  } else {
    // ---------------------------------------------------------------- dQ1, dQ2 / dK1, dK2 epilogue
    const int w4 = warp - 8;
    const int row = w4 * 32 + lane;
    const uint32_t lane_off = uint32_t(w4 * 32) << 16;
    // kBothBoxes 2 KB staging boxes per warp ([32 rows][16 fp32], 64-byte
    // swizzle: 16-byte chunk c of row r at chunk c ^ ((r / 2) % 4)), round
    // robin; dQ1 is read first, dQ2 second, and the accumulator is released
    // after the second read, before that side is staged.
    constexpr int kHalves = D / 32;
    const uint32_t stage = sb + L::oStage + w4 * (kBothBoxes * 2048);
    const uint32_t swz = (lane >> 1) & 3;
    int nred = 0;
    // deterministic mode: every value rounded to its row's grid before it is
    // staged (dq_fixed_exp: mode P1's bound for dQ1, mode P2's for dQ2), so
    // the fp32 reduce-adds are exact in any order; dKL and KL of this
    // thread's row are loaded a tile ahead
    const bool fixed = a.dq_fixed != 0;
    const float kmax1 = fixed ? __uint_as_float(a.kmax[bh] << 16) : 0.f;
    const float kmax2 = fixed ? __uint_as_float(a.kmax[a.BH + bh] << 16) : 0.f;
    float dkl_nx = 0.f, kl_nx = 0.f;
    auto load_row = [&](int i) {
      const int qi = (qt_lo + i) * kTile + row;
      if (fixed && qi < a.NQ && SKL_CHECK(a.status, bh < a.BH)) {
        const size_t idx = size_t(bh) * a.NQ + qi;
        dkl_nx = a.dkl[idx];
        kl_nx = a.kl[idx];
      }
    };
    auto to_grid = [&](uint32_t (&x)[32], float me) {  // (x + me) - me, two values at a time
      const uint64_t ME = f2(me, me);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float q0, q1;
        f2_split(f2_sub(f2_add(f2(__uint_as_float(x[j]), __uint_as_float(x[j + 1])), ME), ME), q0, q1);
        x[j] = __float_as_uint(q0);
        x[j + 1] = __float_as_uint(q1);
      }
    };
    if (n > 0) load_row(0);
    if (lane == 0) {
      tma_prefetch_desc(&tdq1);
      tma_prefetch_desc(&tdq2);
    }
    for (int i = 0; i < n; ++i) {
      if (!mbar_wait_warp(bar(L::B_DQFULL), i & 1, ctl)) break;
      tc_fence_after();
      const int r0 = (qt_lo + i) * kTile + w4 * 32;  // first query row of this warp
      float me[2] = {0.f, 0.f};
      if (fixed) {
        me[0] = 1.5f * exp2_int(23 - dq_fixed_exp(STREAMKL_GRAD_P1, a.scale1, dkl_nx, kl_nx, kmax1));
        me[1] = 1.5f * exp2_int(23 - dq_fixed_exp(STREAMKL_GRAD_P2, a.scale2, dkl_nx, kl_nx, kmax2));
      }
      if (i + 1 < n) load_row(i + 1);
#pragma unroll
      for (int side = 0; side < 2; ++side) {
        uint32_t v[kHalves][32];
#pragma unroll
        for (int x = 0; x < kHalves; ++x) tmem_ld32(t_dq + lane_off + side * 64 + 32 * x, v[x]);
        if (side == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::B_DQEMPTY));
        }
        if (fixed) {
#pragma unroll
          for (int x = 0; x < kHalves; ++x) to_grid(v[x], me[side]);
        }
#pragma unroll
        for (int h = 0; h < 2 * kHalves; ++h) {
          // columns past the head dim (zero-filled operand), or rows all past
          // NQ: no box is touched, so the box count matches the committed
          // reduce groups and no box still being read is overwritten
          if (h * 16 >= a.dg || r0 >= a.NQ) break;
          const uint32_t box = stage + (nred % kBothBoxes) * 2048;
          if (!SKL_CHECK(a.status, box + 2048 <= sb + L::oBar && h * 16 < a.dg)) break;
          if (lane == 0) bulk_wait_read_le<kBothBoxes - 1>();  // the box used kBothBoxes reduces ago was read
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int e = (h & 1) * 16 + 4 * c;
            st_shared_v4(box + lane * 64 + ((c ^ swz) << 4), v[h >> 1][e], v[h >> 1][e + 1], v[h >> 1][e + 2],
                         v[h >> 1][e + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(side == 0 ? &tdq1 : &tdq2, box, h * 16, r0, bh);
            bulk_commit();
          }
          ++nred;
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // every reduce has landed before the CTA exits
    const int kj = k0 + row;
    if (n > 0 && mbar_wait_warp(bar(L::B_DKFULL), 0, ctl)) {
      tc_fence_after();
#pragma unroll
      for (int side = 0; side < 2; ++side) {
        float* dst = (side == 0 ? a.dk : a.dk2) + (size_t(bh) * a.NK + kj) * a.dg;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32((side == 0 ? t_dk1 : t_dk2) + lane_off + ch * 32, v);
          if (kj < a.NK && SKL_CHECK(a.status, bh < a.BH && a.dg <= D)) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              if (ch * 32 + e < a.dg)
                *reinterpret_cast<float4*>(dst + ch * 32 + e) =
                    make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                __uint_as_float(v[e + 3]));
          }
        }
      }
    } else if (n == 0 && kj < a.NK) {
      // no query row sees this key tile: its dK is zero on both sides
      for (int e = 0; e < a.dg; e += 4) {
        *reinterpret_cast<float4*>(a.dk + (size_t(bh) * a.NK + kj) * a.dg + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(a.dk2 + (size_t(bh) * a.NK + kj) * a.dg + e) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D>
static int launch_bwd_both_t(const TMaps& m, const BwdArgs& a, cudaStream_t st) {
  using L = BothLayout<D>;
  auto kern = bwd_both_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid((a.NK + kTile - 1) / kTile, a.BH);
  kern<<<grid, kBothThreads, L::kAlloc, st>>>(m.q1, m.k1, m.q2, m.k2, m.dq, m.dq2, a);
  return cudaGetLastError();
}

int launch_bwd_both(const TMaps& m, int d, const BwdArgs& a, cudaStream_t st) {
  if (d == 64) return launch_bwd_both_t<64>(m, a, st);
  if (d == 32) return launch_bwd_both_t<32>(m, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace skl
