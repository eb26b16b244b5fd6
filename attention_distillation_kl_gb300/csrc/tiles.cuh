// Shared-memory layout of one 128-row bf16 operand tile ([128 rows][D]) as
// the TMA writes it, and its tcgen05 descriptors.
//   D a multiple of 64 (up to 256): D / 64 blocks of [128 rows][64 elements], 128-byte
//                       rows, 128-byte swizzle
//   D = 32:             one block of [128 rows][32 elements], 64-byte rows,
//                       64-byte swizzle
// A descriptor for K-step kk is the step-0 descriptor plus off_k(kk) (the
// tile's rows are K-major, the contraction runs over D in steps of 16) or
// plus off_n(kk) (the tile read as an N-major B operand with N = D, the
// contraction running over its rows in steps of 16).
#pragma once

#include "kernels.cuh"
#include "ptx.cuh"

namespace skl {

template <int D>
struct OpTile {
  static_assert(D == 32 || (D % 64 == 0 && D <= 256), "tile width 32, 64, 128, 192 or 256");
  static constexpr int kD = D;
  static constexpr bool kWide = D >= 64;                 // 128-byte swizzle
  static constexpr int kBox = kWide ? 64 : 32;           // TMA box width, elements
  static constexpr int kBlocks = D / kBox;
  static constexpr uint32_t kBlockBytes = kTile * kBox * 2;
  static constexpr uint32_t kRowBytes = kBox * 2;        // one row of a block
  static constexpr uint32_t kGroup = 8 * kRowBytes;      // 8-row swizzle atom

  __device__ __forceinline__ static uint64_t desc_k(uint32_t base) {
    return kWide ? sdesc_sw128(base, 16, kGroup) : sdesc_sw64(base, 16, kGroup);
  }
  __device__ __forceinline__ static uint32_t off_k(int kk) {
    return (kk / (kBox / 16)) * kBlockBytes + (kk % (kBox / 16)) * 32;
  }
  __device__ __forceinline__ static uint64_t desc_n(uint32_t base) {
    return kWide ? sdesc_sw128(base, kBlockBytes, kGroup) : sdesc_sw64(base, kBlockBytes, kGroup);
  }
  __device__ __forceinline__ static uint32_t off_n(int kk) { return kk * 16 * kRowBytes; }

  // TMA loads of rows [row0, row0 + 128) of head bh into the tile at base.
  __device__ __forceinline__ static void load(uint32_t base, const CUtensorMap* m, uint32_t bar, int row0,
                                              int bh) {
#pragma unroll
    for (int c = 0; c < kBlocks; ++c) tma_load_3d(base + c * kBlockBytes, m, bar, c * kBox, row0, bh);
  }
};

}  // namespace skl
