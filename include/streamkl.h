/*
 * libstreamkl -- fused attention KL divergence on GB300 (sm_103a).
 *
 * For every query row i it computes KL(P1_i || P2_i) with
 *   P1 = softmax(s * Q1 K1^T), P2 = softmax(s * Q2 K2^T)
 * over the visible keys (optionally causal), plus LSE1_i and LSE2_i, without
 * materialising either N_Q x N_K matrix, and the gradient of
 * L = sum_i dKL_i * KL_i with respect to one side's Q and K.
 *
 * Sources: StreamKL article on agidaily.cc, sections "Online formula"
 * (L = acc/l1 + LSE2 - LSE1 with a B_Q-vector rescale of acc), "Forward"
 * (one streaming pass, outputs KL, LSE1, LSE2 only), "Backward" (tile-by-tile
 * recompute of P from the saved LSEs; modes "optimise P2" and "optimise P1"
 * with a numerically stable log-ratio) and "GPU kernel engineering" (key
 * split with a light reduce, fused dQ/dK backward with atomics); and the
 * abstract of "StreamKL: Fast and Memory-Efficient KL Divergence for Boosting
 * Attention Distillation" (arXiv 2606.20005).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout: q1 [B, H, NQ, d1], k1 [B, H, NK, d1], q2 [B, H, NQ, d2],
 *   k2 [B, H, NK, d2], bf16, row-major and contiguous (BHSD).  Per-row
 *   vectors (kl, lse1, lse2, dkl) are fp32 [B, H, NQ], contiguous.
 * Pointers: all tensor pointers are DEVICE pointers on the current device,
 *   16-byte aligned.  The caller owns every buffer (inputs, outputs and the
 *   key-split workspace); the library never allocates, frees or synchronises
 *   and keeps no state between calls other than the device status word.
 * Streams: every call is asynchronous and stream-ordered on `stream`
 *   (a cudaStream_t; NULL = legacy default stream).  Errors detected on the
 *   host return before anything is enqueued.
 * Scale: 0 < scale <= 1e4 and finite; S = scale * Q K^T on both sides (the
 *   *_scaled calls take one scale per side, each under the same rule).
 * Causal: key j is visible to query i iff j <= i + (NK - NQ) (bottom-right
 *   aligned; j <= i when NQ == NK).  causal with NQ > NK is INVALID_ARG.
 * Head dims: d1, d2 any multiple of 16 from 16 to 256, independently
 *   (UNSUPPORTED otherwise).  The kernels compute in tiles 32, 64, 128, 192
 *   or 256 wide; a head dim below its tile width is read with the columns
 *   past it zero-filled, which changes no dot product (the padded work is
 *   not credited in any throughput figure).  Above 128 on either side the
 *   forward streams K in 64-column blocks and the backward always runs as
 *   two passes without atomics (dK, then dQ), whatever `deterministic` says.
 * Empty problems: B*H*NQ == 0 is a no-op that returns OK (the backward then
 *   zeroes dk); NK == 0 with NQ > 0 is INVALID_ARG (rows without keys).
 * Return: a streamkl_status value; C++ exceptions never cross this ABI.
 */
#ifndef STREAMKL_H
#define STREAMKL_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, declared here so users need no CUDA header. */
typedef struct CUstream_st* streamkl_stream_t;

enum streamkl_status {
  STREAMKL_OK = 0,
  STREAMKL_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, causal with NQ > NK, small workspace */
  STREAMKL_UNSUPPORTED = 2,    /* head dim or device not supported */
  STREAMKL_CUDA_ERROR = 3,     /* a CUDA runtime/driver call failed (launch, tensor map, attribute) */
  STREAMKL_DEVICE_TIMEOUT = 4, /* reported by streamkl_get_device_status(): a kernel gave up a wait */
  STREAMKL_DEBUG_BOUNDS = 5    /* reported by streamkl_get_device_status() of a build with STREAMKL_DEBUG
                                  defined: an index a kernel computed failed its bounds check, and the
                                  access was skipped */
};

enum streamkl_grad_mode {
  STREAMKL_GRAD_P2 = 0, /* dS2 = dKL (P2 - P1): gradient into Q2, K2 (head dim d2); standard distillation */
  STREAMKL_GRAD_P1 = 1  /* dS1 = dKL P1 (log P1 - log P2 - KL): gradient into Q1, K1 (head dim d1) */
};

/*
 * Forward: one streaming pass per query tile (article sections "Online
 * formula" and "Forward").  Writes kl, lse1, lse2 (fp32 [B, H, NQ]; natural
 * log).  No buffer beyond the inputs and these outputs is touched.
 */
int streamkl_fwd(const void* q1, const void* k1, const void* q2, const void* k2,
                 int B, int H, int NQ, int NK, int d1, int d2, float scale, int causal,
                 float* kl, float* lse1, float* lse2, streamkl_stream_t stream);

/*
 * Key-split forward (article section "GPU kernel engineering": split along
 * the key dimension when B*H*NQ is too small to fill the GPU, write partial
 * statistics, merge them with a light reduce kernel).  Each of num_splits
 * partitions of every row's visible key tiles writes (m1, l1, acc, m2, l2)
 * to `workspace`; a second kernel merges them into kl, lse1, lse2.
 * workspace: caller-owned device buffer of at least
 *   streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits) bytes, 16-byte
 *   aligned; its contents on entry do not matter and are garbage on return.
 * 1 <= num_splits <= 1024; more splits than key tiles leaves some empty
 * (they contribute nothing).  Results equal streamkl_fwd's up to rounding.
 */
int streamkl_fwd_splitk(const void* q1, const void* k1, const void* q2, const void* k2,
                        int B, int H, int NQ, int NK, int d1, int d2, float scale, int causal,
                        int num_splits, void* workspace, size_t workspace_bytes,
                        float* kl, float* lse1, float* lse2, streamkl_stream_t stream);

/* 5 * 4 * num_splits * B * H * NQ bytes (0 for invalid arguments). */
size_t streamkl_fwd_splitk_workspace_bytes(int B, int H, int NQ, int num_splits);

/*
 * Key-split forward that allocates nothing (the pages have no counterpart:
 * this is an interface for callers, not part of the method).  Some callers
 * cannot call cudaMalloc or hand over a scratch buffer -- for example code
 * inside a framework whose caching allocator owns all device memory, where a
 * raw allocation can synchronise the device and upset its accounting, or a
 * runtime that must not fail for lack of memory in the middle of a step.
 * This variant keeps the per-split partials in one fixed array inside the
 * library: STREAMKL_STATIC_WORKSPACE_BYTES of device memory that every GPU
 * loading the library holds until the process exits.  The caller still
 * passes inputs and outputs exactly as for streamkl_fwd_splitk.
 * Limits: streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits) must not
 *   exceed STREAMKL_STATIC_WORKSPACE_BYTES, else STREAMKL_INVALID_ARG and
 *   nothing is enqueued.
 * Set-up: every call looks the array's device address up afresh (so a
 *   cudaDeviceReset, which reloads the library's module and may move the
 *   array, does no harm); the first call on a device may load the module,
 *   so make it before any stream capture on that device.
 * Sharing: all calls on a device share the array, which keeps the last
 *   call's contents (nothing in it needs to start at zero).  Calls that
 *   overlap on the GPU -- on different streams, or from different host
 *   threads -- race on it; serialise them.
 * No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define STREAMKL_STATIC_WORKSPACE_BYTES ((size_t)32 << 20)
int streamkl_fwd_splitk_noalloc(const void* q1, const void* k1, const void* q2, const void* k2,
                                int B, int H, int NQ, int NK, int d1, int d2, float scale,
                                int causal, int num_splits, float* kl, float* lse1, float* lse2,
                                streamkl_stream_t stream);

/*
 * Advisory split count for the current device: the smallest number of
 * splits that gives at least two waves of CTAs, capped by the key tiles of
 * the longest row.  Returns 1 when no split is needed, 0 on invalid sizes.
 */
int streamkl_suggest_splits(int B, int H, int NQ, int NK, int causal);

/*
 * Backward (article section "Backward"; fused dQ/dK with atomics from
 * "GPU kernel engineering").  Recomputes P1 = exp(S1 - LSE1) and
 * P2 = exp(S2 - LSE2) tile by tile from the forward's kl/lse1/lse2 and the
 * upstream dkl (fp32 [B, H, NQ]), then writes the gradient of
 * sum_i dkl_i * KL_i for the side `mode` selects:
 *   STREAMKL_GRAD_P2: dq = dQ2 [B, H, NQ, d2], dk = dK2 [B, H, NK, d2]
 *   STREAMKL_GRAD_P1: dq = dQ1 [B, H, NQ, d1], dk = dK1 [B, H, NK, d1]
 * dq and dk are fp32 and fully overwritten.  deterministic = 0: one kernel,
 * dq accumulated with fp32 atomics after an on-stream memset (summation order
 * varies run to run).  deterministic = 1: the same kernel, bitwise
 * reproducible: each key tile's contribution to dq row i is rounded to a
 * grid of 2^-e_i before it is added, with 2^-e_i = 2^-22 of a bound on
 * |dQ_i| (from dKL_i, KL_i, the softmax scale and max |K| of the key head),
 * so the fp32 sums are exact in any order; the rounding is at most 2^-22 of
 * that bound per key tile (and at most 2^-127 absolute).  It reads K once
 * more (the bound), and takes a few bytes of scratch (4 per key head of the
 * gradient side, streamkl_bwd_workspace_bytes) from the stream's memory pool
 * (cudaMallocAsync), released on the stream before the call returns;
 * streamkl_bwd_gqa_ws takes it from the caller instead.
 * kl, lse1, lse2 must come from streamkl_fwd on the same inputs.
 */
int streamkl_bwd(const void* q1, const void* k1, const void* q2, const void* k2,
                 int B, int H, int NQ, int NK, int d1, int d2, float scale, int causal,
                 const float* kl, const float* lse1, const float* lse2, const float* dkl,
                 int mode, int deterministic, float* dq, float* dk, streamkl_stream_t stream);

/*
 * Per-side softmax scales: S1 = scale1 * Q1 K1^T and S2 = scale2 * Q2 K2^T,
 * for a student whose head dimension or temperature differs from the
 * teacher's.  (The pages use one scale; a second one is a widening of the
 * method, taken as the plain reading: each softmax keeps its own logits.)
 * Arguments, layout, ownership and errors are those of the single-scale
 * calls, which are these with scale1 = scale2 = scale.  In the backward the
 * gradient side's scale multiplies dQ and dK (s2 in mode P2, s1 in mode P1);
 * kl, lse1, lse2 must come from a forward with the same two scales.
 */
int streamkl_fwd_scaled(const void* q1, const void* k1, const void* q2, const void* k2,
                        int B, int H, int NQ, int NK, int d1, int d2, float scale1, float scale2,
                        int causal, float* kl, float* lse1, float* lse2, streamkl_stream_t stream);
int streamkl_fwd_splitk_scaled(const void* q1, const void* k1, const void* q2, const void* k2,
                               int B, int H, int NQ, int NK, int d1, int d2, float scale1,
                               float scale2, int causal, int num_splits, void* workspace,
                               size_t workspace_bytes, float* kl, float* lse1, float* lse2,
                               streamkl_stream_t stream);
int streamkl_bwd_scaled(const void* q1, const void* k1, const void* q2, const void* k2,
                        int B, int H, int NQ, int NK, int d1, int d2, float scale1, float scale2,
                        int causal, const float* kl, const float* lse1, const float* lse2,
                        const float* dkl, int mode, int deterministic, float* dq, float* dk,
                        streamkl_stream_t stream);

/*
 * Grouped key heads (GQA; MQA with one key head per side).  Not on the
 * pages; taken in the usual sense: q1, q2 have H heads, k1 has HK1 and k2
 * has HK2 heads ([B, HK, NK, d], each count dividing H, else INVALID_ARG),
 * and query head h reads key head h / (H / HK) of its side.  KL, LSE1, LSE2
 * stay per query head [B, H, NQ]; dq is [B, H, NQ, dg]; dk is the gradient
 * of the shared key heads, [B, HK_g, NK, dg] with HK_g the gradient side's
 * count (HK2 in mode P2, HK1 in mode P1): the sum over the query heads
 * that read each key head.  With deterministic = 0 a shared head's dK is
 * added up with fp32 atomics (order not fixed); with deterministic = 1 the
 * query heads of a group add their dK to each key tile in head order (still
 * one launch: a CTA takes its turn from a counter per key head and key
 * tile, which it waits for only when the previous head's CTA for the same
 * key tile is still running), so the result is bitwise repeatable; the
 * counters add 4 bytes per key head and key tile to the scratch block.  Heads
 * above 128 take two passes without atomics (dK, then dQ) whatever
 * `deterministic` says.  Otherwise as the *_scaled calls, which are these
 * with HK1 = HK2 = H.
 */
int streamkl_fwd_gqa(const void* q1, const void* k1, const void* q2, const void* k2,
                     int B, int H, int HK1, int HK2, int NQ, int NK, int d1, int d2,
                     float scale1, float scale2, int causal, float* kl, float* lse1, float* lse2,
                     streamkl_stream_t stream);
int streamkl_fwd_splitk_gqa(const void* q1, const void* k1, const void* q2, const void* k2,
                            int B, int H, int HK1, int HK2, int NQ, int NK, int d1, int d2,
                            float scale1, float scale2, int causal, int num_splits, void* workspace,
                            size_t workspace_bytes, float* kl, float* lse1, float* lse2,
                            streamkl_stream_t stream);
int streamkl_bwd_gqa(const void* q1, const void* k1, const void* q2, const void* k2,
                     int B, int H, int HK1, int HK2, int NQ, int NK, int d1, int d2,
                     float scale1, float scale2, int causal, const float* kl, const float* lse1,
                     const float* lse2, const float* dkl, int mode, int deterministic, float* dq,
                     float* dk, streamkl_stream_t stream);

/*
 * The deterministic backward's scratch from the caller instead of the
 * stream's memory pool, for callers that must not let the library allocate.
 * streamkl_bwd_workspace_bytes returns the bytes it needs: 0 unless
 * deterministic = 1 with both head dims at most 128, else 4 per key head of
 * the gradient side (B * HK_g), 8 more, and 4 per key head and key tile
 * when query heads share key heads (H > HK_g), rounded up to 16; 0 for
 * arguments the backward would reject.  streamkl_bwd_gqa_ws is
 * streamkl_bwd_gqa with `workspace` (device memory, 16-byte aligned, owned
 * by the caller, contents overwritten; may be null when 0 bytes are
 * needed): INVALID_ARG when it is null, misaligned or smaller than needed.
 * The results are bitwise those of streamkl_bwd_gqa.  Calls that overlap on
 * the GPU must not share a workspace.
 */
size_t streamkl_bwd_workspace_bytes(int B, int H, int HK1, int HK2, int NK, int d1, int d2, int mode,
                                    int deterministic);
int streamkl_bwd_gqa_ws(const void* q1, const void* k1, const void* q2, const void* k2,
                        int B, int H, int HK1, int HK2, int NQ, int NK, int d1, int d2,
                        float scale1, float scale2, int causal, const float* kl, const float* lse1,
                        const float* lse2, const float* dkl, int mode, int deterministic, float* dq,
                        float* dk, void* workspace, size_t workspace_bytes, streamkl_stream_t stream);

/*
 * Both-sides backward: the gradients of sum_i dkl_i * KL_i with respect to
 * both distributions (dq1, dk1 with head dim d1; dq2, dk2 with d2; fp32,
 * fully overwritten), from one recompute of S1 and S2 per tile pair when
 * d1 = d2 <= 64.  (A widening of the method: the article's two modes share
 * P1 and P2.)  deterministic = 1 rounds both sides' dQ contributions to
 * their rows' grids as streamkl_bwd does (mode P1's bound for dq1, mode
 * P2's for dq2; scratch of 8 bytes per head from the stream's pool).  Other
 * head-dimension pairs (above 64 the four accumulators do not fit beside S1
 * and S2 in tensor memory; unequal pairs have no one-pass kernel) run the
 * single-side backward twice (mode P2, then mode P1) and return what those
 * return.  Arguments, ownership and errors are otherwise those of
 * streamkl_bwd_scaled; kl, lse1, lse2 must come from a forward with the
 * same two scales.
 */
int streamkl_bwd_both(const void* q1, const void* k1, const void* q2, const void* k2,
                      int B, int H, int NQ, int NK, int d1, int d2, float scale1, float scale2,
                      int causal, const float* kl, const float* lse1, const float* lse2,
                      const float* dkl, int deterministic, float* dq1, float* dk1, float* dq2,
                      float* dk2, streamkl_stream_t stream);

/* Static, NUL-terminated description of a status value. */
const char* streamkl_status_string(int status);

/*
 * Reads and clears the current device's status word.  Kernels bound every
 * wait on an mbarrier (a few seconds); a kernel that gives up sets this word
 * to STREAMKL_DEVICE_TIMEOUT, releases what it holds and exits, leaving its
 * outputs undefined.  Synchronous (it waits for the device).  Returns
 * STREAMKL_OK when no kernel has reported a problem since the last read, or
 * STREAMKL_CUDA_ERROR if the word cannot be read.
 */
int streamkl_get_device_status(void);

/*
 * Self-test of the timeout path (no counterpart on the pages): launches one
 * tiny kernel that waits on a barrier nothing ever completes, gives up after
 * `limit_us` microseconds (1 .. 1e6), sets the device status word to
 * STREAMKL_DEVICE_TIMEOUT and returns; the CUDA context stays usable.  Read
 * the result with streamkl_get_device_status() after synchronising.
 */
int streamkl_selftest_wait_timeout(int limit_us, streamkl_stream_t stream);

/*
 * Self-test of the other bounded wait, the one the deterministic backward
 * uses when query heads share a key head (a CTA waits for a counter in
 * global memory to reach its turn).  `words`: device memory of at least 5
 * ints, 16-byte aligned, owned by the caller and overwritten.  One thread
 * waits for a counter nothing moves; after `limit_us` microseconds (1 ..
 * 1e6) it must give up, set the device status word to
 * STREAMKL_DEVICE_TIMEOUT and set the launch's abort word; a second wait,
 * as another CTA of that launch would make, must then give up at once.
 * Results in words[2..4]: first wait succeeded (0 expected), second wait
 * succeeded (0 expected), second wait returned within a tenth of the limit
 * (1 expected).  Returns INVALID_ARG for a bad limit or pointer.
 */
int streamkl_selftest_turn_timeout(int limit_us, int* words, streamkl_stream_t stream);

/*
 * Device probe used for the roofline denominator: runs `blocks` CTAs of 256
 * threads, each thread evaluating `iters` x 8 independent ex2.approx.f32
 * chains, and writes a checksum to out[0] (device pointer) so the work is
 * not eliminated.  Time it with events on `stream`; rate = blocks * 256 *
 * iters * 8 / time.
 */
int streamkl_probe_ex2(float* out, int blocks, int iters, streamkl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* STREAMKL_H */
