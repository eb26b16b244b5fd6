// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tile loads, tcgen05 (TMEM allocation, MMA, commit, loads) and the shared
// memory matrix descriptors the MMAs read.  Written from the PTX ISA's
// descriptions of these instructions.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "streamkl.h"

namespace skl {

// A kernel abandons a wait after this many nanoseconds of %globaltimer, sets
// the device status word and exits.  Every legitimate wait in these kernels
// lasts micro- to milliseconds.
#ifndef STREAMKL_WAIT_LIMIT_NS
#define STREAMKL_WAIT_LIMIT_NS 4000000000ull
#endif

// Bounds checks of the debug build (compiled with STREAMKL_DEBUG): every
// global-memory index a kernel computes, and the shared-memory staging and
// TMA coordinates, are checked against the extents the kernel was given; a
// failed check skips the access and records STREAMKL_DEBUG_BOUNDS in the
// device status word (no trap, the context stays usable).  In the normal
// build the checks compile to nothing.
#ifdef STREAMKL_DEBUG
#define SKL_CHECK(status, cond) \
  ((cond) ? true : (atomicCAS((status), 0, (int)STREAMKL_DEBUG_BOUNDS), false))
#else
#define SKL_CHECK(status, cond) true
#endif

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Finite stand-in for -inf in running maxima: scaled by any allowed softmax
// scale it stays finite, and its correction factor underflows to exactly 0.
constexpr float kNegBig = -1.0e30f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes in one 64-bit register pair, for the packed FP32 pipe
// instructions (fma/add/sub/mul .rn.f32x2): one issue slot for two values.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Three-input maximum.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared control block of a CTA: the abort flag that every bounded wait polls.
struct Ctl {
  volatile int* abort;  // shared memory
  int* status;          // device status word (global)
};

// Non-blocking probe of the phase with parity `parity`.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Slow path of the bounded wait (kept out of line): polls with try_wait
// until the phase completes, another thread of the CTA aborts, or
// `limit_ns` of %globaltimer pass -- then it aborts the CTA and reports a
// timeout in the status word.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, Ctl ctl,
                                                   uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (*ctl.abort) return false;
    if (globaltimer() - t0 > limit_ns) {
      *ctl.abort = 1;
      atomicCAS(ctl.status, 0, (int)STREAMKL_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// Waits for the phase of `bar` with parity `parity` to complete.  Returns
// false (without waiting further) once any thread of the CTA has aborted;
// after `limit_ns` it aborts the CTA and reports a timeout.  A phase that is
// already complete costs one inline test.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, Ctl ctl, uint64_t limit_ns) {
  if (mbar_test(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, ctl, limit_ns);
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, Ctl ctl) {
  return mbar_wait_limit(bar, parity, ctl, STREAMKL_WAIT_LIMIT_NS);
}

// The same bounded wait without the inline probe: a call straight into the
// polling loop.  Timed faster for the backward's single-thread roles (the
// MMA issuer above all), whose barriers are rarely complete on arrival.
__device__ __forceinline__ bool mbar_wait_polled(uint32_t bar, uint32_t parity, Ctl ctl) {
  return mbar_wait_slow(bar, parity, ctl, STREAMKL_WAIT_LIMIT_NS);
}

// Bounded wait that ignores the abort flag: used on the way out to let copies
// and MMAs that are already in flight land before the CTA releases its
// shared and tensor memory.
static __device__ __noinline__ bool mbar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

// Warp-uniform wait: every lane polls, then the warp agrees; a lane that gave
// up makes the whole warp give up, so .sync.aligned instructions that follow
// are executed by all lanes or none.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, Ctl ctl) {
  bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled load (x = element within a row, y = row, z = batch*head) into
// shared memory, completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// 3-D tiled reduce-add of a shared-memory box into global memory (the
// tensor map's element type, here fp32); rows past the tensor's extent are
// skipped.  Completion is tracked per thread with bulk async-groups.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src, int x, int y,
                                                  int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N committed bulk groups of this thread are still
// reading their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read_le() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (tensor core) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One lane of a converged warp, chosen by elect.sync.  An MMA role that runs
// its loop with all 32 lanes keeps the descriptor arithmetic warp-uniform,
// and only the elected lane issues tcgen05 operations (a role that issues
// from a single-lane branch passes leader = 1).  In a probe, the MMA stream
// issued from a single-lane branch lost up to two thirds of its rate to busy
// warps on the same sub-partition; the converged form kept ~97 %.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t p;
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, e;\n\t}"
      : "=r"(p));
  return p;
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate; issued
// only by the lane whose `leader` is non-zero.
__device__ __forceinline__ void mma_bf16_ss(uint32_t leader, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "setp.ne.b32 q, %4, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation the leader lane issued
// before it has completed.
__device__ __forceinline__ void mma_commit(uint32_t leader, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %1, 0;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
      "r"(leader)
      : "memory");
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major (0 = K, 1 = MN), 16 B major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) |
         (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits 0-13 start >> 4, 16-29 leading byte offset >> 4, 32-45 stride byte
//   offset >> 4, 46-47 version (1), 49-51 base offset (0: atoms are
//   1024-byte aligned), 61-63 layout (2 = 128B swizzle).
// K-major operand stored as [rows][64 bf16] blocks: SBO = 1024 (8-row group
//   stride), LBO unused.  MN-major operand stored as [K rows][64 bf16 of MN]
//   blocks: LBO = stride between 64-element MN blocks, SBO = 1024 (stride
//   between groups of 8 K rows).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// The same descriptor for the 64-byte swizzle (layout 4): K-major operand
// stored as [rows][32 bf16] (64-byte rows): SBO = 512 (8-row group stride);
// MN-major operand stored as [K rows][32 bf16 of MN]: SBO = 512 between
// groups of 8 K rows, LBO = stride between 32-element MN blocks.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(4) << 61;
  return d;
}

// The descriptor of the same operand `bytes` further on: the start address
// field is the low 14 bits (address / 16), and shared-memory addresses stay
// below 2^18, so a plain add never carries out of it.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// Two 32-column loads (32 lanes x 32 bit, one row per thread) and the wait in
// one statement, so no use of the registers can be scheduled before the wait.
#define SKL_R8(a, o) "=r"(a[o + 0]), "=r"(a[o + 1]), "=r"(a[o + 2]), "=r"(a[o + 3]), \
                     "=r"(a[o + 4]), "=r"(a[o + 5]), "=r"(a[o + 6]), "=r"(a[o + 7])

__device__ __forceinline__ void tmem_ld2x32(uint32_t ta, uint32_t tb, uint32_t (&a)[32],
                                            uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : SKL_R8(a, 0), SKL_R8(a, 8), SKL_R8(a, 16), SKL_R8(a, 24), SKL_R8(b, 0), SKL_R8(b, 8),
        SKL_R8(b, 16), SKL_R8(b, 24)
      : "r"(ta), "r"(tb)
      : "memory");
}

// Four 32-column loads and one wait: one round trip to TMEM for a
// warpgroup's 64 columns of both logit matrices.
__device__ __forceinline__ void tmem_ld4x32(uint32_t ta, uint32_t tb, uint32_t tc, uint32_t td,
                                            uint32_t (&a)[32], uint32_t (&b)[32], uint32_t (&c)[32],
                                            uint32_t (&d)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : SKL_R8(a, 0), SKL_R8(a, 8), SKL_R8(a, 16), SKL_R8(a, 24), SKL_R8(b, 0), SKL_R8(b, 8),
        SKL_R8(b, 16), SKL_R8(b, 24), SKL_R8(c, 0), SKL_R8(c, 8), SKL_R8(c, 16), SKL_R8(c, 24),
        SKL_R8(d, 0), SKL_R8(d, 8), SKL_R8(d, 16), SKL_R8(d, 24)
      : "r"(ta), "r"(tb), "r"(tc), "r"(td)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t (&a)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : SKL_R8(a, 0), SKL_R8(a, 8), SKL_R8(a, 16), SKL_R8(a, 24)
      : "r"(ta)
      : "memory");
}

// Moves a whole warpgroup's per-thread register budget down or up (the
// registers one warpgroup gives back are what another can take; an increase
// waits until enough are free, so every decrease must run first or
// concurrently, and the sum over warpgroups must stay within the block's
// launch budget).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace skl
