// Backward kernels: tile-by-tile recompute of P1 = exp(S1 - LSE1) and
// P2 = exp(S2 - LSE2) from the saved log-sum-exps (StreamKL article,
// "Backward"), for the gradient of L = sum_i dKL_i KL_i with respect to one
// side ("optimise P2", the standard distillation case, or "optimise P1"):
//   mode P2:  dS2_ij = dKL_i (P2_ij - P1_ij)
//   mode P1:  dS1_ij = dKL_i P1_ij (r_ij - KL_i),
//             r_ij = (S1_ij - LSE1_i) - (S2_ij - LSE2_i) taken from logits,
//             so nothing is a logarithm of an underflowed probability.
//   dQ = s dS K_g,  dK = s dS^T Q_g  (g = the gradient side; the kernels
//   form s dS before rounding it to bf16, so the products come out scaled).
//
// Fused kernel (article section "GPU kernel engineering": one visit per
// query/key tile pair, dQ through atomics).  One CTA owns a 128-key tile and
// walks the query tiles that can see it.  GB300 mapping, 15 or 16 warps:
//   warp 12    TMA: K1, K2 once; per query tile Q_o (single buffer) and Q_g
//              (two or three buffers; it is read again by the dK product)
//   warp 13    TMEM owner, S issuer:
//                S1 = Q1 K1^T, S2 = Q2 K2^T      (M = queries, N = keys)
//   warp 14    dK issuer:   dK += dS^T Q_g       (accumulates in TMEM)
//              and, in mode P2, dQ = dS K_g      (per query tile)
//   warp 15    mode P1 only: dQ issuer
//              Separate issuing threads, so no product waits behind another's
//              barriers (S of tile i+1 runs while dS of tile i is formed).
//   warps 0-7  thread = query row: P1/P2 and dS from S (TMEM) with the
//              row's LSE/dKL/KL in registers (loaded one tile ahead);
//              warps 0-3 take key columns 0-63, warps 4-7 columns 64-127
//              (two warps per SM sub-partition, and S is released after
//              half the work).  dS goes to shared memory as bf16 rows in the
//              128-byte-swizzled layout both products read: K-major A for
//              dQ, M-major A (dS^T) for dK
//   warps 8-11 dQ tile: TMEM -> registers (96 columns, one box staged, the
//              last 32 columns, then the accumulator is free; the register
//              budget of 512 threads holds no whole 128-column row)
//              -> 32 x 32 fp32 boxes in 128-byte-swizzled
//              shared memory (two per warp, round robin) -> TMA bulk tensor
//              reduce-add into global dQ (rows past NQ are clipped by the
//              tensor map); finally dK (stored; when several query heads
//              share a key head, added with atomics, or in the deterministic
//              mode in head order, see wait_turn)
// TMEM: S1 [0,128), S2 [128,256), dK [256, 256+dg), dQ [384, 384+dg).
//
// Deterministic mode: the same kernel, with each dQ contribution rounded to
// a per-row grid of 2^-e before the reduce-add, fine enough to keep the row's
// precision and coarse enough that the fp32 sums are exact in whatever
// order they land (bound and grid: dq_fixed_exp; max |K| per key head:
// dq_fixed.cu); dK is written by one CTA anyway.
#include "bwd_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace skl {


constexpr int kDqBoxes = 2;          // dQ staging boxes per epilogue warp
constexpr uint32_t kDqBoxBytes = 4096;  // [32 rows][32 fp32], 128-byte swizzle

template <int D1, int D2, int MODE>
struct BwdLayout {
  static constexpr int DG = MODE == STREAMKL_GRAD_P2 ? D2 : D1;  // gradient side
  static constexpr int DO = MODE == STREAMKL_GRAD_P2 ? D1 : D2;  // other side
  // Mode P1 forms dS with one ex2 per pair, so the MMA issue chain is what
  // bounds it: dK and dQ then get an issuing thread each (16 warps).  In
  // mode P2 the dS warps bound the tile and one thread issues both (15).
  static constexpr bool kSplitIssue = MODE == STREAMKL_GRAD_P1;
  static constexpr int kThreads = 32 * (kSplitIssue ? 16 : 15);
  static constexpr uint32_t kDS = kTile * kTile * 2;
  static constexpr uint32_t kK1 = kTile * D1 * 2, kK2 = kTile * D2 * 2;
  static constexpr uint32_t kQo = kTile * DO * 2, kQg = kTile * DG * 2;
  enum {
    B_KFULL, B_QOFULL, B_QOEMPTY, B_QGFULL0, B_QGFULL1, B_QGFULL2, B_QGEMPTY0, B_QGEMPTY1, B_QGEMPTY2,
    B_SFULL, B_SFREE, B_DSFULL, B_DSEMPTY, B_DQFULL, B_DQEMPTY, B_DKFULL, B_DONE, kNumBars
  };
  // Q_g buffers: its buffer of tile t is free again only when the dK
  // product of tile t has run, and that product comes late in the tile (it
  // waits for dS and for the next tile's S to be queued), so two buffers
  // chain the reload of tile t + 2 to the dK of tile t; a third buffer,
  // where it fits (every pair of head dims but 128 and 128), takes the
  // reload off that chain
  static constexpr uint32_t kFixed = kDS + kK1 + kK2 + kQo + 4 * kDqBoxes * kDqBoxBytes + kNumBars * 8 + 32;
  static constexpr int kQgBufs = kFixed + 3 * kQg + 1024 <= 232448 ? 3 : 2;
  static constexpr uint32_t oDS = 0, oK1 = kDS, oK2 = oK1 + kK1, oQo = oK2 + kK2, oQg = oQo + kQo;
  static constexpr uint32_t oStage = oQg + kQgBufs * kQg;  // dQ staging: 4 warps x kDqBoxes x kDqBoxBytes
  static constexpr uint32_t oBar = oStage + 4 * kDqBoxes * kDqBoxBytes;
  static constexpr uint32_t oMisc = oBar + kNumBars * 8;
  static constexpr uint32_t kBytes = oMisc + 32;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "over the 227 KB shared memory limit");
};

// The gradient products of tile t are issued only once the S products of
// tile t + 1 are queued: the tensor pipe takes them in issue order, and S is
// what the dS warps wait for, so S should not queue behind dK and dQ.  A
// scheduling hint only (the two groups touch different TMEM columns and
// operands), so the wait gives up after 20 us rather than reporting anything.
__device__ __forceinline__ void wait_s_queued(volatile int* s_queued, int want) {
  if (want <= 0 || *s_queued >= want) return;
  const uint64_t t0 = globaltimer();
  while (*s_queued < want && globaltimer() - t0 < 20000ull) {
  }
}

// Grouped key heads, deterministic mode: waits until the count of query
// heads that have added their dK to this (key head, key tile) reads `want`,
// polling with a short sleep.  Gives up when this CTA or another one has
// aborted, or after `limit_ns`; then this CTA aborts, and a time-out also
// aborts the launch and is reported in the status word.
static __device__ __noinline__ bool wait_turn(const int* turn, int want, int* launch_abort, Ctl ctl,
                                              uint64_t limit_ns = STREAMKL_WAIT_LIMIT_NS) {
  const uint64_t t0 = globaltimer();
  while (true) {
    if (ld_acquire_gpu(turn) == want) return true;
    if (*ctl.abort || *reinterpret_cast<volatile int*>(launch_abort)) {
      *ctl.abort = 1;
      return false;
    }
    if (globaltimer() - t0 > limit_ns) {
      *ctl.abort = 1;
      atomicExch(launch_abort, 1);
      atomicCAS(ctl.status, 0, (int)STREAMKL_DEVICE_TIMEOUT);
      return false;
    }
    __nanosleep(128);
  }
}

template <int D1, int D2, int MODE>
__global__ void __launch_bounds__(BwdLayout<D1, D2, MODE>::kThreads, 1)
    bwd_fused_kernel(const __grid_constant__ CUtensorMap tq1, const __grid_constant__ CUtensorMap tk1,
                     const __grid_constant__ CUtensorMap tq2, const __grid_constant__ CUtensorMap tk2,
                     const __grid_constant__ CUtensorMap tdq, const BwdArgs a) {
  using L = BwdLayout<D1, D2, MODE>;
  constexpr int DG = L::DG, DO = L::DO;
  constexpr bool kP2 = MODE == STREAMKL_GRAD_P2;
  using T1 = OpTile<D1>;
  using T2 = OpTile<D2>;
  using TO = OpTile<DO>;
  using TG = OpTile<DG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int gg = kP2 ? a.g2 : a.g1;  // query heads per gradient-side key head

  auto bar = [&](int id) { return sb + L::oBar + 8u * id; };
  const CUtensorMap* tqo = kP2 ? &tq1 : &tq2;
  const CUtensorMap* tqg = kP2 ? &tq2 : &tq1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oMisc + 4);
  // query tiles whose S products the S issuer has queued (a scheduling
  // hint for the gradient issuers, see below)
  volatile int* s_queued = reinterpret_cast<volatile int*>(smem + L::oMisc + 8);
  int* unit_slot = reinterpret_cast<int*>(smem + L::oMisc + 12);
  volatile int* turn_ok = reinterpret_cast<volatile int*>(smem + L::oMisc + 16);
  const Ctl ctl{abort_flag, a.status};

  if (threadIdx.x == 0) {
    // ordered dK of grouped key heads: units (key tile fastest, then query
    // head; head_group is 1) in the order CTAs start, so a head waits only
    // for CTAs that run
    *unit_slot = a.ticket ? atomicAdd(a.ticket, 1) : int(blockIdx.y * gridDim.x + blockIdx.x);
    *s_queued = 0;
    for (int b = 0; b < L::kNumBars; ++b) {
      uint32_t count = 1;  // TMA transaction barriers and tcgen05.commit targets
      if (b == L::B_SFREE || b == L::B_DSFULL) count = 8;  // one per dS warp
      if (b == L::B_DQEMPTY) count = 4;                    // one per epilogue warp
      if (b == L::B_DSEMPTY) count = L::kSplitIssue ? 2 : 1;  // dK (and dQ) issuers
      if (b == L::B_DONE) count = L::kSplitIssue ? 3 : 2;  // one per MMA issuer
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
  const uint32_t t_s1 = tmem, t_s2 = tmem + 128, t_dk = tmem + 256, t_dq = tmem + 384;

  // unit -> (query head (batch-major), key tile): heads in groups of
  // head_group whose key tiles interleave, the longest sweeps first
  int bh, kt;
  grouped_unit(*unit_slot, a.BH, int(gridDim.x), a.head_group, bh, kt);
  const int k0 = kt * kTile;
  const int off = a.NK - a.NQ;
  const int nqt = (a.NQ + kTile - 1) / kTile;
  // causal: query i sees key j iff i >= j - off; the first query tile that
  // sees any key of this tile starts at row max(0, k0 - off)
  const int qt_lo = a.causal ? max(0, k0 - off) / kTile : 0;
  const int n = nqt - qt_lo;

  if (warp == 12) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tq1);
      tma_prefetch_desc(&tk1);
      tma_prefetch_desc(&tq2);
      tma_prefetch_desc(&tk2);
      mbar_arrive_expect_tx(bar(L::B_KFULL), L::kK1 + L::kK2);
      T1::load(sb + L::oK1, &tk1, bar(L::B_KFULL), k0, bh / a.g1);
      T2::load(sb + L::oK2, &tk2, bar(L::B_KFULL), k0, bh / a.g2);
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int q0 = (qt_lo + i) * kTile;
        if (!mbar_wait_polled(bar(L::B_QOEMPTY), (i & 1) ^ 1, ctl)) break;
        mbar_arrive_expect_tx(bar(L::B_QOFULL), L::kQo);
        TO::load(sb + L::oQo, tqo, bar(L::B_QOFULL), q0, bh);
        const int g = i % L::kQgBufs;
        if (!mbar_wait_polled(bar(L::B_QGEMPTY0 + g), ((i / L::kQgBufs) & 1) ^ 1, ctl)) break;
        mbar_arrive_expect_tx(bar(L::B_QGFULL0 + g), L::kQg);
        TG::load(sb + L::oQg + g * L::kQg, tqg, bar(L::B_QGFULL0 + g), q0, bh);
        issued = i + 1;
      }
      if (*abort_flag) {  // let the copies already started land before the CTA exits
        const uint64_t lim = 200000000ull;
        mbar_drain(bar(L::B_KFULL), 0, lim);
        if (issued > 0) mbar_drain(bar(L::B_QOFULL), (issued - 1) & 1, lim);
        for (int i = issued > L::kQgBufs ? issued - L::kQgBufs : 0; i < issued; ++i)
          mbar_drain(bar(L::B_QGFULL0 + i % L::kQgBufs), (i / L::kQgBufs) & 1, lim);
      }
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------------- S issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);
      // S of one side for query tile i: Q tile (A, K-major) x K (B, K-major)
      auto s_product = [&](auto tile, uint32_t d, uint32_t qs, uint32_t ks) {
        using T = decltype(tile);
        const uint64_t qd = T::desc_k(qs), kd = T::desc_k(ks);
#pragma unroll
        for (int kk = 0; kk < T::kD / 16; ++kk) {
          const uint32_t o = T::off_k(kk);
          mma_bf16_ss(1u, d, sdesc_add(qd, o), sdesc_add(kd, o), id_s, kk > 0);
        }
      };
      bool ok = n > 0 && mbar_wait_polled(bar(L::B_KFULL), 0, ctl);
      for (int i = 0; ok && i < n; ++i) {
        if (!mbar_wait_polled(bar(L::B_SFREE), (i & 1) ^ 1, ctl)) break;
        if (!mbar_wait_polled(bar(L::B_QOFULL), i & 1, ctl)) break;
        tc_fence_after();
        // the other side first: its single Q buffer is released as early as possible
        if constexpr (kP2) s_product(T1{}, t_s1, sb + L::oQo, sb + L::oK1);
        else s_product(T2{}, t_s2, sb + L::oQo, sb + L::oK2);
        mma_commit(1u, bar(L::B_QOEMPTY));
        if (!mbar_wait_polled(bar(L::B_QGFULL0 + i % L::kQgBufs), (i / L::kQgBufs) & 1, ctl)) break;
        tc_fence_after();
        if constexpr (kP2) s_product(T2{}, t_s2, sb + L::oQg + (i % L::kQgBufs) * L::kQg, sb + L::oK2);
        else s_product(T1{}, t_s1, sb + L::oQg + (i % L::kQgBufs) * L::kQg, sb + L::oK1);
        mma_commit(1u, bar(L::B_SFULL));
        *s_queued = i + 1;
      }
      // every MMA of every issuer has finished before TMEM is released
      mma_commit(1u, bar(L::B_DONE));
      mbar_drain(bar(L::B_DONE), 0, 1000000000ull);
    }
  } else if (warp == 14) {
    // ---------------------------------------------------------------- dK (and dQ) issuer
    if (lane == 0) {
      constexpr bool kDq = !L::kSplitIssue;  // this thread also issues dQ
      constexpr uint32_t id_dk = idesc_bf16(128, DG, 1, 1);  // A = dS^T M-major, B = Q_g N-major
      constexpr uint32_t id_dq = idesc_bf16(128, DG, 0, 1);  // A = dS K-major,   B = K_g N-major
      const uint64_t dsm = sdesc_sw128(sb + L::oDS, kTile * 128, 1024);  // dS^T, M-major
      const uint64_t dsk = sdesc_sw128(sb + L::oDS, 16, 1024);           // dS, K-major
      const uint64_t kgn = TG::desc_n(sb + (kP2 ? L::oK2 : L::oK1));
      int t = 0;
      if (n > 0 && mbar_wait_polled(bar(L::B_KFULL), 0, ctl)) {
        for (; t < n; ++t) {
          if (!mbar_wait_polled(bar(L::B_DSFULL), t & 1, ctl)) break;
          wait_s_queued(s_queued, t + 1 < n ? t + 2 : 0);
          tc_fence_after();
          const uint64_t qgn = TG::desc_n(sb + L::oQg + (t % L::kQgBufs) * L::kQg);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss(1u, t_dk, sdesc_add(dsm, kk * 2048), sdesc_add(qgn, TG::off_n(kk)), id_dk,
                        (t > 0 || kk > 0) ? 1u : 0u);
          mma_commit(1u, bar(L::B_QGEMPTY0 + t % L::kQgBufs));  // Q_g(t) may be reloaded
          if (kDq) {
            // dK and the Q_g release above did not wait for the dQ accumulator
            if (!mbar_wait_polled(bar(L::B_DQEMPTY), (t & 1) ^ 1, ctl)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_bf16_ss(1u, t_dq, sdesc_add(dsk, (kk >> 2) * (kTile * 128) + (kk & 3) * 32),
                          sdesc_add(kgn, TG::off_n(kk)), id_dq, kk > 0 ? 1u : 0u);
          }
          mma_commit(1u, bar(L::B_DSEMPTY));
          if (kDq) mma_commit(1u, bar(L::B_DQFULL));
        }
      }
      if (n > 0 && t == n && !*abort_flag) mma_commit(1u, bar(L::B_DKFULL));
      mma_commit(1u, bar(L::B_DONE));  // the TMEM owner drains it before releasing TMEM
    }
  } else if (warp == 15) {  // exists in mode P1 only
    if constexpr (L::kSplitIssue) {
      // ---------------------------------------------------------------- dQ issuer (mode P1)
      if (lane == 0) {
        constexpr uint32_t id_dq = idesc_bf16(128, DG, 0, 1);  // A = dS K-major, B = K_g N-major
        const uint64_t dsk = sdesc_sw128(sb + L::oDS, 16, 1024);  // dS, K-major
        const uint64_t kgn = TG::desc_n(sb + (kP2 ? L::oK2 : L::oK1));
        if (n > 0 && mbar_wait_polled(bar(L::B_KFULL), 0, ctl)) {
          for (int t = 0; t < n; ++t) {
            if (!mbar_wait_polled(bar(L::B_DSFULL), t & 1, ctl)) break;
            wait_s_queued(s_queued, t + 1 < n ? t + 2 : 0);
            if (!mbar_wait_polled(bar(L::B_DQEMPTY), (t & 1) ^ 1, ctl)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_bf16_ss(1u, t_dq, sdesc_add(dsk, (kk >> 2) * (kTile * 128) + (kk & 3) * 32),
                          sdesc_add(kgn, TG::off_n(kk)), id_dq, kk > 0 ? 1u : 0u);
            mma_commit(1u, bar(L::B_DSEMPTY));
            mma_commit(1u, bar(L::B_DQFULL));
          }
        }
        mma_commit(1u, bar(L::B_DONE));  // the TMEM owner drains it before releasing TMEM
      }
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------- dS (thread = query row)
    // warpgroup wg takes key columns [64 wg, 64 wg + 64) of every tile
    const int wg = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float c1 = a.scale1 * kLog2e, c2 = a.scale2 * kLog2e, nr = -a.scale2 / a.scale1;
    const uint64_t C1 = f2(c1, c1), C2 = f2(c2, c2), S1 = f2(a.scale1, a.scale1), NR = f2(nr, nr);
    const float sg = kP2 ? a.scale2 : a.scale1;  // softmax scale of the gradient side
    // per-row parameters of query tile i (see ds_chunk_row)
    auto params = [&](int i, float& na, float& nb, float& ws) {
      const int qi = (qt_lo + i) * kTile + row;
      na = -INFINITY;
      nb = kP2 ? -INFINITY : 0.f;
      ws = 0.f;
      if (qi < a.NQ && SKL_CHECK(a.status, bh < a.BH)) {
        const size_t idx = size_t(bh) * a.NQ + qi;
        const float l1 = a.lse1[idx];
        na = -l1 * kLog2e;
        ws = sg * a.dkl[idx];
        nb = kP2 ? -a.lse2[idx] * kLog2e : -(l1 - a.lse2[idx] + a.kl[idx]);
      }
    };
    float na, nb, ws;
    if (n > 0) params(0, na, nb, ws);
    for (int i = 0; i < n; ++i) {
      const int q0 = (qt_lo + i) * kTile;
      const uint64_t NA = f2(na, na), NB = f2(nb, nb), WW = f2(ws, ws);
      if (i + 1 < n) params(i + 1, na, nb, ws);  // used next tile: the loads overlap this one
      if (!mbar_wait_warp(bar(L::B_SFULL), i & 1, ctl)) break;
      tc_fence_after();
      // last visible key of this row, relative to the tile
      const int lim = (a.causal ? min(q0 + row + off, a.NK - 1) : a.NK - 1) - k0;
      const bool need_mask = (k0 + kTile > a.NK) || (a.causal && q0 < k0 + kTile - 1 - off);
      uint32_t dsr[32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int col = wg * 64 + ch * 32;
        uint32_t x1[32], x2[32];
        tmem_ld2x32(t_s1 + lane_off + col, t_s2 + lane_off + col, x1, x2);
        if (ch == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::B_SFREE));
        }
        if (need_mask)
          ds_chunk_row<MODE, true>(x1, x2, C1, C2, S1, NR, NA, NB, WW, lim - col, dsr + ch * 16);
        else
          ds_chunk_row<MODE, false>(x1, x2, C1, C2, S1, NR, NA, NB, WW, 0, dsr + ch * 16);
      }
      // the previous tile's products must be done reading dS before it is replaced
      if (!mbar_wait_warp(bar(L::B_DSEMPTY), (i & 1) ^ 1, ctl)) break;
      store_half_row_sw128(sb + L::oDS, row, wg, dsr);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_DSFULL));
    }
  } else {
    // ---------------------------------------------------------------- dQ / dK epilogue
    const int w4 = warp - 8;
    const int row = w4 * 32 + lane;
    const uint32_t lane_off = uint32_t(w4 * 32) << 16;
    {
      // This thread's dQ row (DG fp32) is read from TMEM and the accumulator
      // released before most of it is staged, so the next dQ product rarely
      // waits for the reduce-adds.  The row leaves in boxes of [32 rows][32 fp32]
      // (128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8); one
      // full 128-byte line per row) through kDqBoxes staging boxes per warp,
      // each a bulk tensor reduce-add into the fp32 dQ.  For dg = 16 the map
      // has boxes of [32 rows][16 fp32] with the 64-byte swizzle instead
      // (chunk c of row r at c ^ ((r / 2) % 4)).  In the deterministic mode
      // the row is first rounded to its grid of 2^-e (dq_fixed_exp), so the
      // fp32 sums are exact in any order.
      constexpr int kChunks = DG / 32;
      const bool wide = a.dq_box == 32;
      const uint32_t stage = sb + L::oStage + w4 * (kDqBoxes * kDqBoxBytes);
      int nred = 0;
      if (lane == 0) tma_prefetch_desc(&tdq);
      const bool fixed = a.dq_fixed != 0;
      const float sg = kP2 ? a.scale2 : a.scale1;
      const float kmax = fixed ? __uint_as_float(a.kmax[bh / gg] << 16) : 0.f;
      // deterministic mode: dKL and KL of this thread's row in query tile i
      // (the row's grid), loaded a tile ahead
      float dkl_nx = 0.f, kl_nx = 0.f;
      auto load_row = [&](int i) {
        const int qi = (qt_lo + i) * kTile + row;
        if (fixed && qi < a.NQ && SKL_CHECK(a.status, bh < a.BH)) {
          const size_t idx = size_t(bh) * a.NQ + qi;
          dkl_nx = a.dkl[idx];
          kl_nx = a.kl[idx];
        }
      };
      // each value rounded to the row's grid of 2^-e: (x + 1.5 * 2^(23 - e))
      // - 1.5 * 2^(23 - e), two values at a time on the FMA pipe
      auto to_fixed = [&](uint32_t (&x)[32], uint64_t ME) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float q0, q1;
          f2_split(f2_sub(f2_add(f2(__uint_as_float(x[j]), __uint_as_float(x[j + 1])), ME), ME), q0, q1);
          x[j] = __float_as_uint(q0);
          x[j + 1] = __float_as_uint(q1);
        }
      };
      if (n > 0) load_row(0);
      for (int i = 0; i < n; ++i) {
        if (!mbar_wait_warp(bar(L::B_DQFULL), i & 1, ctl)) break;
        tc_fence_after();
        const int r0 = (qt_lo + i) * kTile + w4 * 32;  // first query row of this warp
        const float me = fixed ? 1.5f * exp2_int(23 - dq_fixed_exp(MODE, sg, dkl_nx, kl_nx, kmax)) : 0.f;
        const uint64_t ME = f2(me, me);
        if (i + 1 < n) load_row(i + 1);
        uint32_t v[kChunks][32];
        // one box of the dQ tile: row `lane` of this warp's 32 rows, columns [32 h, 32 h + 32)
        auto put_box = [&](int h) {
          // columns past the head dim (zero-filled operand), or rows all past
          // NQ: nothing to add, and no box is touched (the box count must
          // match the committed reduce groups, or a box still being read by
          // an earlier reduce could be overwritten)
          if (h * 32 >= a.dg || r0 >= a.NQ) return;
          const uint32_t box = stage + (nred % kDqBoxes) * kDqBoxBytes;
          if (!SKL_CHECK(a.status, box + kDqBoxBytes <= sb + L::oBar && h * 32 < a.dg && r0 < a.NQ)) return;
          // the box used kDqBoxes reduces ago has been read
          if (lane == 0) bulk_wait_read_le<kDqBoxes - 1>();
          __syncwarp();
          if (wide) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_shared_v4(box + lane * 128 + ((c ^ (lane & 7)) << 4), v[h][4 * c], v[h][4 * c + 1],
                           v[h][4 * c + 2], v[h][4 * c + 3]);
          } else {
            const uint32_t swz = (lane >> 1) & 3;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              st_shared_v4(box + lane * 64 + ((c ^ swz) << 4), v[h][4 * c], v[h][4 * c + 1], v[h][4 * c + 2],
                           v[h][4 * c + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tdq, box, h * 32, r0, bh);
            bulk_commit();
          }
          ++nred;
        };
        // read the tile; at DG = 128 the first box is staged before the last
        // 32 columns are read, so at most 96 columns are live at once
        if constexpr (kChunks == 4) {
          tmem_ld2x32(t_dq + lane_off, t_dq + lane_off + 32, v[0], v[1]);
          tmem_ld32(t_dq + lane_off + 64, v[2]);
          if (fixed) to_fixed(v[0], ME);
          put_box(0);
          tmem_ld32(t_dq + lane_off + 96, v[3]);
        } else if constexpr (kChunks == 2) {
          tmem_ld2x32(t_dq + lane_off, t_dq + lane_off + 32, v[0], v[1]);
        } else {
          tmem_ld32(t_dq + lane_off, v[0]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::B_DQEMPTY));
#pragma unroll
        for (int h = kChunks == 4 ? 1 : 0; h < kChunks; ++h) {
          if (fixed) to_fixed(v[h], ME);
          put_box(h);
        }
      }
      if (lane == 0) bulk_wait_all();  // every reduce has landed before the CTA exits
    }
    // dK of key head bh / gg: stored, or (grouped key heads) added to what
    // the other query heads of the group contribute
    const int kj = k0 + row;
    float* dst = a.dk + (size_t(bh / gg) * a.NK + kj) * a.dg;
    auto write_dk = [&](int how) {
#pragma unroll
      for (int ch = 0; ch < DG / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(t_dk + lane_off + ch * 32, v);
        if (kj < a.NK && SKL_CHECK(a.status, bh / gg < a.BH / gg && a.dg <= DG)) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            if (ch * 32 + e < a.dg)
              put_dk4(dst + ch * 32 + e,
                      make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                  __uint_as_float(v[e + 3])),
                      how);
        }
      }
    };
    auto zero_dk = [&]() {  // no query row sees this key tile
      if (kj < a.NK)
        for (int e = 0; e < a.dg; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    };
    if (a.dk_turns == nullptr) {
      const int dk_how = gg == 1 ? kDkStore : kDkAtomic;  // atomics: a shared key head, any order
      if (n > 0 && mbar_wait_warp(bar(L::B_DKFULL), 0, ctl)) {
        tc_fence_after();
        write_dk(dk_how);
      } else if (n == 0 && dk_how == kDkStore) {
        zero_dk();
      }
    } else {
      // Deterministic, grouped key heads: the query heads of a group add in
      // head order.  Head m of the group waits until the (key head, key
      // tile) count reads m, then stores (m = 0) or adds, and the count
      // moves on once all four warps' rows are written.  Every epilogue
      // warp reaches both barriers whatever happened (each wait before them
      // is bounded); the count is not moved by a CTA that gave up.
      const int member = bh % gg;
      int* turn = a.dk_turns + size_t(bh / gg) * gridDim.x + kt;
      const bool have = n > 0 && mbar_wait_warp(bar(L::B_DKFULL), 0, ctl);
      if (warp == 8 && lane == 0) *turn_ok = wait_turn(turn, member, a.dk_abort, ctl) ? 1 : 0;
      named_bar_sync(1, 128);
      if (*turn_ok) {
        if (have) {
          tc_fence_after();
          write_dk(member == 0 ? kDkStore : kDkAdd);
        } else if (n == 0 && member == 0) {
          zero_dk();
        }
      }
      named_bar_sync(1, 128);
      if (warp == 8 && lane == 0) {
        if (*turn_ok && !*abort_flag) {
          __threadfence();
          st_release_gpu(turn, member + 1);
        } else {
          atomicExch(a.dk_abort, 1);
        }
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

template <int D1, int D2, int MODE>
static int launch_fused_t(const TMaps& m, const BwdArgs& a, cudaStream_t st) {
  using L = BwdLayout<D1, D2, MODE>;
  auto kern = bwd_fused_kernel<D1, D2, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid((a.NK + kTile - 1) / kTile, a.BH);
  kern<<<grid, L::kThreads, L::kAlloc, st>>>(m.q1, m.k1, m.q2, m.k2, m.dqw, a);
  return cudaGetLastError();
}

// Self-test of the turn wait (one thread, no fault): words = {count, launch
// abort, out[0..2]}, zeroed.  Waits for a count nothing moves, which must
// give up after limit_ns, report a time-out and set the launch abort word;
// then, as another CTA would, waits again, which must give up at once on
// the abort word.  out = {first wait returned, second returned, second
// gave up within a tenth of the limit}.
__global__ void turn_selftest_kernel(int* words, int* status, uint64_t limit_ns) {
  __shared__ int abort_flag;
  abort_flag = 0;
  Ctl ctl{&abort_flag, status};
  words[2] = wait_turn(words, 1, words + 1, ctl, limit_ns) ? 1 : 0;
  abort_flag = 0;
  const uint64_t t0 = globaltimer();
  words[3] = wait_turn(words, 1, words + 1, ctl, limit_ns) ? 1 : 0;
  words[4] = globaltimer() - t0 < limit_ns / 10 ? 1 : 0;
}

int launch_turn_selftest(int* words, int* status, uint64_t limit_ns, cudaStream_t st) {
  turn_selftest_kernel<<<1, 1, 0, st>>>(words, status, limit_ns);
  return cudaGetLastError();
}

#define SKL_DISPATCH_CASE(FN, A, B) \
  if (d1 == A && d2 == B) return p2 ? FN<A, B, 0>(m, a, st) : FN<A, B, 1>(m, a, st);
#define SKL_DISPATCH(FN)                                                                     \
  do {                                                                                       \
    const bool p2 = a.mode == STREAMKL_GRAD_P2;                                              \
    SKL_DISPATCH_CASE(FN, 128, 128) SKL_DISPATCH_CASE(FN, 128, 64) SKL_DISPATCH_CASE(FN, 128, 32) \
    SKL_DISPATCH_CASE(FN, 64, 128) SKL_DISPATCH_CASE(FN, 64, 64) SKL_DISPATCH_CASE(FN, 64, 32)    \
    SKL_DISPATCH_CASE(FN, 32, 128) SKL_DISPATCH_CASE(FN, 32, 64) SKL_DISPATCH_CASE(FN, 32, 32)    \
    return cudaErrorInvalidValue;                                                            \
  } while (0)

int launch_bwd_fused(const TMaps& m, int d1, int d2, const BwdArgs& a, cudaStream_t st) {
  SKL_DISPATCH(launch_fused_t);
}

}  // namespace skl
