// C-ABI entry points of libstreamkl: argument validation, TMA tensor maps,
// launches.  Every check that can fail does so before anything is enqueued.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "streamkl.h"

namespace {

// The device status word that kernels set when they give up a wait.
__device__ int g_status;

int* status_ptr() {
  int* p = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_status) != cudaSuccess) return nullptr;
  return p;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// The kernels' tile width for head dim d (a multiple of 16 up to 256): 32,
// 64, 128, 192 or 256.  Columns past d in a tile are zero-filled by the TMA, which
// leaves every dot product unchanged.
int tile_dim(int d) { return d <= 32 ? 32 : (d <= 64 ? 64 : (d <= 128 ? 128 : (d <= 192 ? 192 : 256))); }

// [BH][N][d] bf16 viewed as a 3-D tensor; boxes of 64 elements x 128 rows x 1
// with the 128-byte swizzle, or for tile width 32 one box of 32 elements x
// 128 rows x 1 with the 64-byte swizzle (the layouts the kernels' operand
// tiles expect).  Rows past N and columns past d read as zeros.
bool make_map(CUtensorMap* m, const void* ptr, long long BH, long long N, int d) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(N), cuuint64_t(BH)};
  cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(N) * d * 2};
  const bool narrow = tile_dim(d) == 32;
  cuuint32_t box[3] = {narrow ? 32u : 64u, cuuint32_t(skl::kTile), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// dQ [BH][NQ][dg] fp32 as a 3-D tensor: boxes of 16 elements x 32 rows x 1,
// 64-byte swizzle, the target of the backward's bulk reduce-adds.
bool make_map_dq(CUtensorMap* m, void* ptr, long long BH, long long NQ, int dg) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {cuuint64_t(dg), cuuint64_t(NQ), cuuint64_t(BH)};
  cuuint64_t strides[2] = {cuuint64_t(dg) * 4, cuuint64_t(NQ) * dg * 4};
  cuuint32_t box[3] = {16, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The fused backward's dQ target: boxes of 32 fp32 x 32 rows with the
// 128-byte swizzle (one full 128-byte line per row and box: fewer, larger
// reduce operations than 64-byte pieces), or the 16-wide map for dg = 16.
bool make_map_dq_wide(CUtensorMap* m, void* ptr, long long BH, long long NQ, int dg, int* box_cols) {
  if (dg < 32) {
    *box_cols = 16;
    return make_map_dq(m, ptr, BH, NQ, dg);
  }
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {cuuint64_t(dg), cuuint64_t(NQ), cuuint64_t(BH)};
  cuuint64_t strides[2] = {cuuint64_t(dg) * 4, cuuint64_t(NQ) * dg * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  *box_cols = 32;
  return r == CUDA_SUCCESS;
}

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f && s <= 1.0e4f; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool head_dim_ok(int d) { return d >= 16 && d <= 256 && d % 16 == 0; }

// Shared validation of the problem description.  Returns STREAMKL_OK, or the
// status to report.  Sets *empty when there is no row to compute.
int check_problem(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H, int HK1,
                  int HK2, int NQ, int NK, int d1, int d2, float scale, int causal, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || NQ < 0 || NK < 0) return STREAMKL_INVALID_ARG;
  // key heads: each side's count divides the query head count
  if (HK1 < 0 || HK2 < 0 || HK1 > H || HK2 > H) return STREAMKL_INVALID_ARG;
  if (H > 0 && (HK1 == 0 || HK2 == 0 || H % HK1 != 0 || H % HK2 != 0)) return STREAMKL_INVALID_ARG;
  if (!scale_ok(scale)) return STREAMKL_INVALID_ARG;
  if (causal != 0 && causal != 1) return STREAMKL_INVALID_ARG;
  if (!head_dim_ok(d1) || !head_dim_ok(d2)) return STREAMKL_UNSUPPORTED;
  if (causal && NQ > NK) return STREAMKL_INVALID_ARG;
  const long long BH = (long long)B * H;
  if (BH == 0 || NQ == 0) {
    *empty = true;
    return STREAMKL_OK;
  }
  if (NK == 0) return STREAMKL_INVALID_ARG;
  // grid.y carries B*H; per-row indices must stay in int range
  if (BH > 65535 || BH * (long long)(NQ > NK ? NQ : NK) > (1ll << 31) - 1) return STREAMKL_INVALID_ARG;
  if (!q1 || !k1 || !q2 || !k2) return STREAMKL_INVALID_ARG;
  if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2)) return STREAMKL_INVALID_ARG;
  return STREAMKL_OK;
}

int device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STREAMKL_CUDA_ERROR;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return STREAMKL_CUDA_ERROR;
  if (major != 10 || minor != 3) return STREAMKL_UNSUPPORTED;  // built for sm_103a only
  return STREAMKL_OK;
}

int make_maps(skl::TMaps* m, const void* q1, const void* k1, const void* q2, const void* k2, int B, int H,
              int HK1, int HK2, int NQ, int NK, int d1, int d2) {
  if (!make_map(&m->q1, q1, (long long)B * H, NQ, d1) || !make_map(&m->k1, k1, (long long)B * HK1, NK, d1) ||
      !make_map(&m->q2, q2, (long long)B * H, NQ, d2) || !make_map(&m->k2, k2, (long long)B * HK2, NK, d2))
    return STREAMKL_CUDA_ERROR;
  return STREAMKL_OK;
}

int as_status(int cuda_err) { return cuda_err == 0 ? STREAMKL_OK : STREAMKL_CUDA_ERROR; }

// Heads whose CTAs interleave (FwdArgs::head_group): as many as keep the
// operand every CTA of a head re-reads (`bytes_per_head`: K for the
// forward; Q and the fp32 dQ for the backward) within a quarter of L2, so
// that interleaving the heads' longest tiles first costs no extra DRAM
// traffic.  (Half of L2 let two heads of 64K tokens share it, 32 MB of K
// each, and the forward then read 1 GB more from DRAM.)
int head_group_for(int BH, double bytes_per_head) {
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
    return 1;
  const double g = 0.25 * double(l2) / (bytes_per_head > 1.0 ? bytes_per_head : 1.0);
  return g < 1.0 ? 1 : (g >= double(BH) ? BH : int(g));
}

}  // namespace

extern "C" {

int streamkl_fwd_gqa(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H, int HK1,
                     int HK2, int NQ, int NK, int d1, int d2, float scale1, float scale2, int causal, float* kl,
                     float* lse1, float* lse2, streamkl_stream_t stream) {
  bool empty = false;
  int s = check_problem(q1, k1, q2, k2, B, H, HK1, HK2, NQ, NK, d1, d2, scale1, causal, &empty);
  if (s == STREAMKL_OK && !scale_ok(scale2)) s = STREAMKL_INVALID_ARG;
  if (s != STREAMKL_OK || empty) return s;
  if (!kl || !lse1 || !lse2 || !aligned16(kl) || !aligned16(lse1) || !aligned16(lse2))
    return STREAMKL_INVALID_ARG;
  if ((s = device_ok()) != STREAMKL_OK) return s;
  skl::TMaps m{};
  if ((s = make_maps(&m, q1, k1, q2, k2, B, H, HK1, HK2, NQ, NK, d1, d2)) != STREAMKL_OK) return s;
  int* st = status_ptr();
  if (!st) return STREAMKL_CUDA_ERROR;
  skl::FwdArgs a{B * H, NQ, NK, causal, 1, H / HK1, H / HK2, scale1, scale2, kl, lse1, lse2, nullptr, st};
  a.head_group = head_group_for(B * H, 2.0 * NK * (d1 + d2));
  return as_status(skl::launch_fwd(m, tile_dim(d1), tile_dim(d2), a, reinterpret_cast<cudaStream_t>(stream)));
}

int streamkl_fwd_scaled(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H,
                        int NQ, int NK, int d1, int d2, float scale1, float scale2, int causal, float* kl,
                        float* lse1, float* lse2, streamkl_stream_t stream) {
  return streamkl_fwd_gqa(q1, k1, q2, k2, B, H, H, H, NQ, NK, d1, d2, scale1, scale2, causal, kl, lse1, lse2,
                          stream);
}

int streamkl_fwd(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H,
                 int NQ, int NK, int d1, int d2, float scale, int causal, float* kl, float* lse1,
                 float* lse2, streamkl_stream_t stream) {
  return streamkl_fwd_scaled(q1, k1, q2, k2, B, H, NQ, NK, d1, d2, scale, scale, causal, kl, lse1, lse2,
                             stream);
}

size_t streamkl_fwd_splitk_workspace_bytes(int B, int H, int NQ, int num_splits) {
  if (B < 0 || H < 0 || NQ < 0 || num_splits < 1 || num_splits > 1024) return 0;
  return size_t(5) * 4 * size_t(num_splits) * size_t(B) * size_t(H) * size_t(NQ);
}

int streamkl_fwd_splitk_gqa(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H,
                            int HK1, int HK2, int NQ, int NK, int d1, int d2, float scale1, float scale2,
                            int causal, int num_splits, void* workspace, size_t workspace_bytes, float* kl,
                            float* lse1, float* lse2, streamkl_stream_t stream) {
  bool empty = false;
  int s = check_problem(q1, k1, q2, k2, B, H, HK1, HK2, NQ, NK, d1, d2, scale1, causal, &empty);
  if (s == STREAMKL_OK && !scale_ok(scale2)) s = STREAMKL_INVALID_ARG;
  if (s != STREAMKL_OK) return s;
  if (num_splits < 1 || num_splits > 1024) return STREAMKL_INVALID_ARG;
  if (empty) return STREAMKL_OK;
  if (!kl || !lse1 || !lse2 || !aligned16(kl) || !aligned16(lse1) || !aligned16(lse2))
    return STREAMKL_INVALID_ARG;
  const size_t need = streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return STREAMKL_INVALID_ARG;
  if ((s = device_ok()) != STREAMKL_OK) return s;
  skl::TMaps m{};
  if ((s = make_maps(&m, q1, k1, q2, k2, B, H, HK1, HK2, NQ, NK, d1, d2)) != STREAMKL_OK) return s;
  int* st = status_ptr();
  if (!st) return STREAMKL_CUDA_ERROR;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(workspace);
  skl::FwdArgs a{B * H, NQ, NK, causal, num_splits, H / HK1, H / HK2, scale1, scale2, kl, lse1, lse2, part, st};
  a.head_group = head_group_for(B * H, 2.0 * NK * (d1 + d2));
  int e = skl::launch_fwd(m, tile_dim(d1), tile_dim(d2), a, cs);
  if (e != 0) return STREAMKL_CUDA_ERROR;
  return as_status(skl::launch_splitk_reduce(part, B * H * NQ, num_splits, kl, lse1, lse2, cs));
}

int streamkl_fwd_splitk_scaled(const void* q1, const void* k1, const void* q2, const void* k2, int B,
                               int H, int NQ, int NK, int d1, int d2, float scale1, float scale2, int causal,
                               int num_splits, void* workspace, size_t workspace_bytes, float* kl,
                               float* lse1, float* lse2, streamkl_stream_t stream) {
  return streamkl_fwd_splitk_gqa(q1, k1, q2, k2, B, H, H, H, NQ, NK, d1, d2, scale1, scale2, causal, num_splits,
                                 workspace, workspace_bytes, kl, lse1, lse2, stream);
}

int streamkl_fwd_splitk(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H,
                        int NQ, int NK, int d1, int d2, float scale, int causal, int num_splits,
                        void* workspace, size_t workspace_bytes, float* kl, float* lse1, float* lse2,
                        streamkl_stream_t stream) {
  return streamkl_fwd_splitk_scaled(q1, k1, q2, k2, B, H, NQ, NK, d1, d2, scale, scale, causal, num_splits,
                                    workspace, workspace_bytes, kl, lse1, lse2, stream);
}

int streamkl_suggest_splits(int B, int H, int NQ, int NK, int causal) {
  if (B <= 0 || H <= 0 || NQ <= 0 || NK <= 0 || (causal != 0 && causal != 1) || (causal && NQ > NK)) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return 1;  // no device to size for: no split
  const long long nqt = (NQ + skl::kTile - 1) / skl::kTile;
  const long long ctas = (long long)B * H * nqt;
  if (ctas >= 4ll * sms) return 1;  // several waves of whole rows already
  const int max_kt = (NK + skl::kTile - 1) / skl::kTile;
  const int off = NK - NQ;
  // Cost model in units of one key tile of one CTA: a CTA with t key tiles
  // takes t + kFixed (Q load, pipeline fill, epilogue); the CTAs (one per SM,
  // longest first) finish after max(total / SMs, longest CTA); a split count
  // s > 1 adds the merge kernel (a launch plus 20 bytes per row and split).
  constexpr double kFixed = 3.0, kMergeLaunch = 10.0, kMergeBytesPerTile = 3.6e6;
  const double rows = double(B) * H * NQ;
  int best = 1;
  double best_t = 0.0;
  for (int s = 1; s <= 1024 && s <= max_kt; ++s) {
    double total = 0.0, longest = 0.0;
    for (long long qt = 0; qt < nqt; ++qt) {
      const long long kend = causal ? (long long)std::min<long long>((qt + 1) * skl::kTile, NQ) + off : NK;
      const long long tiles = (kend + skl::kTile - 1) / skl::kTile;
      // splits take contiguous shares of the key tiles; the largest share bounds the CTA
      const double t = double((tiles + s - 1) / s) + kFixed;
      total += t * s;
      longest = std::max(longest, t);
    }
    total *= double(B) * H;
    double t = std::max(total / sms, longest);
    if (s > 1) t += kMergeLaunch + rows * s * 20.0 / kMergeBytesPerTile;
    if (s == 1 || t < best_t * 0.98) {  // a split has to earn its merge
      best = s;
      best_t = t;
    }
  }
  return best;
}

size_t streamkl_bwd_workspace_bytes(int B, int H, int HK1, int HK2, int NK, int d1, int d2, int mode,
                                    int deterministic) {
  if (B < 0 || H < 0 || NK < 0 || HK1 <= 0 || HK2 <= 0 || H % HK1 != 0 || H % HK2 != 0) return 0;
  if (mode != STREAMKL_GRAD_P2 && mode != STREAMKL_GRAD_P1) return 0;
  if (deterministic != 1 || !head_dim_ok(d1) || !head_dim_ok(d2)) return 0;
  if (tile_dim(d1) > 128 || tile_dim(d2) > 128) return 0;  // the wide-head passes need none
  const int hkg = mode == STREAMKL_GRAD_P2 ? HK2 : HK1;
  const size_t kg_heads = size_t(B) * hkg;
  const size_t key_tiles = (size_t(NK) + skl::kTile - 1) / skl::kTile;
  const size_t words = kg_heads + 2 + (H / hkg > 1 ? kg_heads * key_tiles : 0);
  return (words * 4 + 15) / 16 * 16;
}

}  // extern "C"

namespace {

// The backward behind both entry points.  caller_ws: the scratch of a
// deterministic call is the caller's `workspace` (checked against
// streamkl_bwd_workspace_bytes); otherwise it comes from the stream's memory
// pool and goes back to it on the stream.
int bwd_impl(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H, int HK1, int HK2,
             int NQ, int NK, int d1, int d2, float scale1, float scale2, int causal, const float* kl,
             const float* lse1, const float* lse2, const float* dkl, int mode, int deterministic, float* dq,
             float* dk, bool caller_ws, void* workspace, size_t workspace_bytes, streamkl_stream_t stream) {
  bool empty = false;
  int s = check_problem(q1, k1, q2, k2, B, H, HK1, HK2, NQ, NK, d1, d2, scale1, causal, &empty);
  if (s == STREAMKL_OK && !scale_ok(scale2)) s = STREAMKL_INVALID_ARG;
  if (s != STREAMKL_OK) return s;
  if (mode != STREAMKL_GRAD_P2 && mode != STREAMKL_GRAD_P1) return STREAMKL_INVALID_ARG;
  if (deterministic != 0 && deterministic != 1) return STREAMKL_INVALID_ARG;
  const int dg = mode == STREAMKL_GRAD_P2 ? d2 : d1;
  const int hkg = mode == STREAMKL_GRAD_P2 ? HK2 : HK1;  // key heads of dk
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t dk_bytes = size_t(B) * hkg * NK * dg * 4;
  if (empty) {
    // no query rows: dK is zero (dq is empty)
    if (dk_bytes == 0) return STREAMKL_OK;
    if (!dk || !aligned16(dk)) return STREAMKL_INVALID_ARG;
    return as_status(cudaMemsetAsync(dk, 0, dk_bytes, cs));
  }
  if (!kl || !lse1 || !lse2 || !dkl || !dq || !dk) return STREAMKL_INVALID_ARG;
  if (!aligned16(kl) || !aligned16(lse1) || !aligned16(lse2) || !aligned16(dkl) || !aligned16(dq) ||
      !aligned16(dk))
    return STREAMKL_INVALID_ARG;
  if ((s = device_ok()) != STREAMKL_OK) return s;
  skl::TMaps m{};
  if ((s = make_maps(&m, q1, k1, q2, k2, B, H, HK1, HK2, NQ, NK, d1, d2)) != STREAMKL_OK) return s;
  int* st = status_ptr();
  if (!st) return STREAMKL_CUDA_ERROR;
  const int gg = H / hkg;  // query heads per key head of dk
  skl::BwdArgs a{B * H, NQ, NK, causal, mode, dg, H / HK1, H / HK2, -1, scale1, scale2, kl, lse1, lse2, dkl, dq,
                 dk, st};
  const int t1 = tile_dim(d1), t2 = tile_dim(d2);
  if (t1 > 128 || t2 > 128) {
    // a head above 128: dK by key tiles (the launches of a key-head group in
    // order, the first storing), then dQ by query tiles; no atomics, so both
    // values of `deterministic` take this path
    // (CTA order: heads interleaved in groups that keep the re-read Q, then
    // K, of a group within a quarter of L2)
    a.head_group = head_group_for(B * H, 2.0 * NQ * (d1 + d2));
    for (int j = 0; j < gg; ++j) {
      a.hsel = gg > 1 ? j : -1;
      if (skl::launch_bwd_wide_pass0(m, t1, t2, a, cs) != 0) return STREAMKL_CUDA_ERROR;
    }
    a.hsel = -1;
    a.head_group = head_group_for(B * H, 2.0 * NK * (d1 + d2));
    return as_status(skl::launch_bwd_wide_pass1(m, t1, t2, a, cs));
  }
  // CTA order: heads interleave in groups within L2's reach (not with the
  // ordered dK of the deterministic grouped-head mode: there the query
  // heads of a key-head group would reach the same key tile together and
  // wait on each other's dK, 3-14 % slower than head after head)
  a.head_group = head_group_for(B * H, 2.0 * NQ * (d1 + d2) + 4.0 * NQ * dg);
  if (!deterministic) {
    const size_t dq_bytes = size_t(B) * H * NQ * dg * 4;
    if (!make_map_dq_wide(&m.dqw, dq, (long long)B * H, NQ, dg, &a.dq_box)) return STREAMKL_CUDA_ERROR;
    if (cudaMemsetAsync(dq, 0, dq_bytes, cs) != cudaSuccess) return STREAMKL_CUDA_ERROR;
    // a shared key head's dK is accumulated by the CTAs of its query heads
    if (gg > 1 && cudaMemsetAsync(dk, 0, dk_bytes, cs) != cudaSuccess) return STREAMKL_CUDA_ERROR;
    return as_status(skl::launch_bwd_fused(m, t1, t2, a, cs));
  }
  // deterministic: the same fused kernel in one launch, with every dQ
  // contribution rounded to its row's grid (fp32 sums exact in any order)
  // and, when query heads share a key head, their dK added in head order
  // (the first stores).  Scratch, one block: the bound on |K| per key head,
  // then the launch's ticket and abort word, then one dK count per (key
  // head, key tile) when heads share key heads.
  const size_t dq_bytes = size_t(B) * H * NQ * dg * 4;
  const size_t kg_heads = size_t(B) * hkg;
  const size_t ws_bytes = streamkl_bwd_workspace_bytes(B, H, HK1, HK2, NK, d1, d2, mode, 1);
  if (caller_ws && (workspace == nullptr || !aligned16(workspace) || workspace_bytes < ws_bytes))
    return STREAMKL_INVALID_ARG;
  if (!make_map_dq_wide(&m.dqw, dq, (long long)B * H, NQ, dg, &a.dq_box)) return STREAMKL_CUDA_ERROR;
  if (cudaMemsetAsync(dq, 0, dq_bytes, cs) != cudaSuccess) return STREAMKL_CUDA_ERROR;
  unsigned* scratch = caller_ws ? static_cast<unsigned*>(workspace) : nullptr;
  const bool pooled = !caller_ws;
  if (pooled && cudaMallocAsync(reinterpret_cast<void**>(&scratch), ws_bytes, cs) != cudaSuccess)
    return STREAMKL_CUDA_ERROR;
  int rc = STREAMKL_OK;
  if (cudaMemsetAsync(scratch, 0, ws_bytes, cs) != cudaSuccess ||
      skl::launch_kmax(mode == STREAMKL_GRAD_P2 ? k2 : k1, int(kg_heads), NK, dg, scratch, cs) != 0)
    rc = STREAMKL_CUDA_ERROR;
  a.dq_fixed = 1;
  a.kmax = scratch;
  if (gg > 1) {
    int* words_i = reinterpret_cast<int*>(scratch);
    a.head_group = 1;
    a.ticket = words_i + kg_heads;
    a.dk_abort = words_i + kg_heads + 1;
    a.dk_turns = words_i + kg_heads + 2;
  }
  if (rc == STREAMKL_OK && skl::launch_bwd_fused(m, t1, t2, a, cs) != 0) rc = STREAMKL_CUDA_ERROR;
  if (pooled && cudaFreeAsync(scratch, cs) != cudaSuccess) rc = STREAMKL_CUDA_ERROR;
  return rc;
}

}  // namespace

extern "C" {

int streamkl_bwd_gqa(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H, int HK1,
                     int HK2, int NQ, int NK, int d1, int d2, float scale1, float scale2, int causal,
                     const float* kl, const float* lse1, const float* lse2, const float* dkl, int mode,
                     int deterministic, float* dq, float* dk, streamkl_stream_t stream) {
  return bwd_impl(q1, k1, q2, k2, B, H, HK1, HK2, NQ, NK, d1, d2, scale1, scale2, causal, kl, lse1, lse2, dkl,
                  mode, deterministic, dq, dk, false, nullptr, 0, stream);
}

int streamkl_bwd_gqa_ws(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H, int HK1,
                        int HK2, int NQ, int NK, int d1, int d2, float scale1, float scale2, int causal,
                        const float* kl, const float* lse1, const float* lse2, const float* dkl, int mode,
                        int deterministic, float* dq, float* dk, void* workspace, size_t workspace_bytes,
                        streamkl_stream_t stream) {
  return bwd_impl(q1, k1, q2, k2, B, H, HK1, HK2, NQ, NK, d1, d2, scale1, scale2, causal, kl, lse1, lse2, dkl,
                  mode, deterministic, dq, dk, true, workspace, workspace_bytes, stream);
}

int streamkl_bwd_scaled(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H,
                        int NQ, int NK, int d1, int d2, float scale1, float scale2, int causal,
                        const float* kl, const float* lse1, const float* lse2, const float* dkl, int mode,
                        int deterministic, float* dq, float* dk, streamkl_stream_t stream) {
  return streamkl_bwd_gqa(q1, k1, q2, k2, B, H, H, H, NQ, NK, d1, d2, scale1, scale2, causal, kl, lse1, lse2,
                          dkl, mode, deterministic, dq, dk, stream);
}

int streamkl_bwd(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H,
                 int NQ, int NK, int d1, int d2, float scale, int causal, const float* kl,
                 const float* lse1, const float* lse2, const float* dkl, int mode, int deterministic,
                 float* dq, float* dk, streamkl_stream_t stream) {
  return streamkl_bwd_scaled(q1, k1, q2, k2, B, H, NQ, NK, d1, d2, scale, scale, causal, kl, lse1, lse2, dkl,
                             mode, deterministic, dq, dk, stream);
}

int streamkl_bwd_both(const void* q1, const void* k1, const void* q2, const void* k2, int B, int H, int NQ,
                      int NK, int d1, int d2, float scale1, float scale2, int causal, const float* kl,
                      const float* lse1, const float* lse2, const float* dkl, int deterministic, float* dq1,
                      float* dk1, float* dq2, float* dk2, streamkl_stream_t stream) {
  bool empty = false;
  int s = check_problem(q1, k1, q2, k2, B, H, H, H, NQ, NK, d1, d2, scale1, causal, &empty);
  if (s == STREAMKL_OK && !scale_ok(scale2)) s = STREAMKL_INVALID_ARG;
  if (s != STREAMKL_OK) return s;
  if (deterministic != 0 && deterministic != 1) return STREAMKL_INVALID_ARG;
  if (d1 != d2 || tile_dim(d1) > 64 || empty) {
    // one recompute per side (the single-side kernels; they also handle empty problems)
    s = streamkl_bwd_scaled(q1, k1, q2, k2, B, H, NQ, NK, d1, d2, scale1, scale2, causal, kl, lse1, lse2,
                            dkl, STREAMKL_GRAD_P2, deterministic, dq2, dk2, stream);
    if (s != STREAMKL_OK) return s;
    return streamkl_bwd_scaled(q1, k1, q2, k2, B, H, NQ, NK, d1, d2, scale1, scale2, causal, kl, lse1, lse2,
                               dkl, STREAMKL_GRAD_P1, deterministic, dq1, dk1, stream);
  }
  if (!kl || !lse1 || !lse2 || !dkl || !dq1 || !dk1 || !dq2 || !dk2) return STREAMKL_INVALID_ARG;
  if (!aligned16(kl) || !aligned16(lse1) || !aligned16(lse2) || !aligned16(dkl) || !aligned16(dq1) ||
      !aligned16(dk1) || !aligned16(dq2) || !aligned16(dk2))
    return STREAMKL_INVALID_ARG;
  if ((s = device_ok()) != STREAMKL_OK) return s;
  skl::TMaps m{};
  if ((s = make_maps(&m, q1, k1, q2, k2, B, H, H, H, NQ, NK, d1, d2)) != STREAMKL_OK) return s;
  if (!make_map_dq(&m.dq, dq1, (long long)B * H, NQ, d1) || !make_map_dq(&m.dq2, dq2, (long long)B * H, NQ, d1))
    return STREAMKL_CUDA_ERROR;
  int* st = status_ptr();
  if (!st) return STREAMKL_CUDA_ERROR;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t dq_bytes = size_t(B) * H * NQ * d1 * 4;
  if (cudaMemsetAsync(dq1, 0, dq_bytes, cs) != cudaSuccess || cudaMemsetAsync(dq2, 0, dq_bytes, cs) != cudaSuccess)
    return STREAMKL_CUDA_ERROR;
  skl::BwdArgs a{B * H, NQ, NK, causal, STREAMKL_GRAD_P2, d1, 1, 1, -1, scale1, scale2, kl, lse1, lse2,
                 dkl, dq1, dk1, st, dq2, dk2};
  a.head_group = head_group_for(B * H, 12.0 * NQ * d1);  // Q1, Q2 and both fp32 dQ
  if (!deterministic) return as_status(skl::launch_bwd_both(m, tile_dim(d1), a, cs));
  // deterministic: both dQ sides on their rows' grids (dK is stored by one
  // CTA per key tile anyway); the bound on |K| of both sides' key heads in
  // a scratch block from the stream's pool
  const size_t kbytes = size_t(2) * B * H * sizeof(unsigned);
  unsigned* kmax = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&kmax), kbytes, cs) != cudaSuccess) return STREAMKL_CUDA_ERROR;
  int rc = STREAMKL_OK;
  if (cudaMemsetAsync(kmax, 0, kbytes, cs) != cudaSuccess ||
      skl::launch_kmax(k1, B * H, NK, d1, kmax, cs) != 0 ||
      skl::launch_kmax(k2, B * H, NK, d2, kmax + size_t(B) * H, cs) != 0)
    rc = STREAMKL_CUDA_ERROR;
  a.dq_fixed = 1;
  a.kmax = kmax;
  if (rc == STREAMKL_OK && skl::launch_bwd_both(m, tile_dim(d1), a, cs) != 0) rc = STREAMKL_CUDA_ERROR;
  if (cudaFreeAsync(kmax, cs) != cudaSuccess) rc = STREAMKL_CUDA_ERROR;
  return rc;
}

const char* streamkl_status_string(int status) {
  switch (status) {
    case STREAMKL_OK: return "ok";
    case STREAMKL_INVALID_ARG: return "invalid argument";
    case STREAMKL_UNSUPPORTED: return "unsupported head dimension or device";
    case STREAMKL_CUDA_ERROR: return "CUDA error";
    case STREAMKL_DEVICE_TIMEOUT: return "a kernel abandoned a wait (device timeout)";
    case STREAMKL_DEBUG_BOUNDS: return "debug build: an index failed its bounds check (access skipped)";
    default: return "unknown status";
  }
}

int streamkl_get_device_status(void) {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return STREAMKL_CUDA_ERROR;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return STREAMKL_CUDA_ERROR;
  return v;
}

int streamkl_selftest_wait_timeout(int limit_us, streamkl_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return STREAMKL_INVALID_ARG;
  int s = device_ok();
  if (s != STREAMKL_OK) return s;
  int* st = status_ptr();
  if (!st) return STREAMKL_CUDA_ERROR;
  return as_status(skl::launch_wait_selftest(st, uint64_t(limit_us) * 1000u,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int streamkl_selftest_turn_timeout(int limit_us, int* words, streamkl_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000 || !words || !aligned16(words)) return STREAMKL_INVALID_ARG;
  int s = device_ok();
  if (s != STREAMKL_OK) return s;
  int* st = status_ptr();
  if (!st) return STREAMKL_CUDA_ERROR;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(words, 0, 5 * sizeof(int), cs) != cudaSuccess) return STREAMKL_CUDA_ERROR;
  return as_status(skl::launch_turn_selftest(words, st, uint64_t(limit_us) * 1000u, cs));
}

int streamkl_probe_ex2(float* out, int blocks, int iters, streamkl_stream_t stream) {
  if (!out || blocks < 1 || iters < 1 || blocks > (1 << 20)) return STREAMKL_INVALID_ARG;
  return as_status(skl::launch_ex2_probe(out, blocks, iters, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
