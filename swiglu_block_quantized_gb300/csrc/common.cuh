// common.cuh -- inline-PTX building blocks for sm_103a: mbarriers with
// time-bounded waits, TMA tile loads, and tcgen05 (TMEM alloc, MMA, ld/st).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace m4q {

// Codec ids (same values as enum m4q_codec in include/m4q.h).
enum : int { kQ4_0 = 0, kQ8_0 = 1, kQ2_0 = 2, kMLX4 = 3 };

// Status-word bits: a bounded wait gave up; a bounds check failed (only in
// the bounds-checked build, below).
enum : uint32_t { kErrWaitTimeout = 1u, kErrAborted = 2u, kErrBounds = 4u };

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ bounds
//
// The bounds-checked build (-DM4Q_BOUNDS=1) tests each computed global
// access, each TMA coordinate and each computed shared-memory staging offset
// against the extents the kernel knows, before making the access.  A failed
// test sets kErrBounds in status word 0, records its site number in word 2
// (the first failure only) and the access is skipped, so a wrong index is
// reported instead of faulting.  (A skipped copy leaves its barrier short:
// the bounded wait behind it then gives up and is reported as well.)  In the
// normal build every test is the constant true.
#ifndef M4Q_BOUNDS
#define M4Q_BOUNDS 0
#endif

enum : uint32_t {
  kSiteGemvW = 1,        // GEMV: bulk copy of a weight row pair
  kSiteGemvWHalf = 2,    // GEMV: 2-byte weight copy into the ring
  kSiteGemvX = 3,        // GEMV: activation fragment load
  kSiteGemvY = 4,        // GEMV: output store
  kSiteTcX = 5,          // tcgen05 kernels: X tile coordinates
  kSiteTcW = 6,          // tcgen05 kernels: packed-W tile coordinates
  kSiteTcY = 7,          // tcgen05 kernels: Y tile coordinates
  kSiteTcWRow = 8,       // tcgen05 kernels: packed row read from the W ring
  kSiteTcStage = 9,      // tcgen05 kernels: Y staging offset
  kSiteTcSplitSlot = 10, // K split: staged partial offset
  kSiteTcSplitY = 11,    // K split: output store
  kSiteTcBRing = 12,     // small-M kernel: decoded-B ring offset
  kSiteAttnQ = 20,       // attention: Q fragment load
  kSiteAttnKV = 21,      // attention: K/V tile copy
  kSiteAttnO = 22,       // attention: output store
  kSiteAttnWs = 23,      // attention: key-split workspace
};

__device__ __forceinline__ bool in_bounds(bool cond, uint32_t* status, uint32_t site) {
#if M4Q_BOUNDS
  if (!cond) {
    atomicOr(status, kErrBounds);
    atomicCAS(status + 2, 0u, site);
  }
  return cond;
#else
  (void)status;
  (void)site;
  return true;
#endif
}

// [off, off + bytes) inside [0, size)
__device__ __forceinline__ bool span_ok(long long off, long long bytes, long long size) {
  return off >= 0 && bytes >= 0 && off + bytes <= size;
}

// A tiled TMA copy starts on a 16-byte boundary: the innermost coordinate
// times the element size is a multiple of 16; no coordinate of a store may
// be negative.
__device__ __forceinline__ bool tma_x_ok(int x, int elem_bytes) { return x >= 0 && (x * elem_bytes) % 16 == 0; }

// First byte of `base` (dynamic shared memory) aligned to `A` bytes.  The
// pointer is advanced, not rebuilt from an integer, so the compiler still
// knows it addresses shared memory and emits shared-memory loads and stores
// for everything derived from it (a pointer rebuilt from an integer is
// generic: every access then goes through a 64-bit generic address).
template <uint32_t A>
__device__ __forceinline__ uint8_t* smem_align(uint8_t* base) {
  return base + ((A - (smem_u32(base) & (A - 1))) & (A - 1));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// GELU(g) = g * Phi(g) = g/2 * erfc(-g / sqrt 2), in fp32 (the GeGLU gate).
__device__ __forceinline__ float gelu_f(float g) { return 0.5f * g * erfcf(-g * 0.70710678118654752f); }

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// One arrival per warp: the lanes meet at a warp barrier first, so every
// lane's earlier writes (and, after a proxy fence, its async-proxy-visible
// shared-memory writes) are ordered before the arrival.  Barriers that a
// whole warp signals count warps, not threads: per-thread arrivals on one
// barrier serialize in shared memory.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared abort state of one CTA: once any thread gives up, the rest stop
// waiting at their next poll instead of each running out its own limit.
struct WaitCtl {
  volatile int* abort;   // shared-memory flag
  uint32_t* status;      // device status word (global)
  uint64_t limit_ns;     // per-wait limit
};

// Slow path of mbar_wait: poll until the phase completes, the limit passes or
// another thread of the CTA has given up.  Never spins without bound.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*ctl.abort) return false;
      if (global_timer_ns() - t0 > ctl.limit_ns) {
        *ctl.abort = 1;
        atomicOr(ctl.status, kErrWaitTimeout);
        return false;
      }
    }
  }
}

// Slow path of mbar_wait_idle: like mbar_wait_slow, but the thread sleeps
// between polls (32 ns doubling up to max_ns), so a warp that waits a long
// time leaves the issue slots of its SM sub-partition to the working warps.
static __device__ __noinline__ bool mbar_wait_idle_slow(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                                        uint32_t max_ns) {
  const uint64_t t0 = global_timer_ns();
  uint32_t ns = 32;
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*ctl.abort) return false;
    if (global_timer_ns() - t0 > ctl.limit_ns) {
      *ctl.abort = 1;
      atomicOr(ctl.status, kErrWaitTimeout);
      return false;
    }
    __nanosleep(ns);
    if (ns < max_ns) ns *= 2;
  }
}

// Wait for `bar` to complete the phase with the given parity.  Returns false
// (after recording the failure) if the limit passes or another thread of the
// CTA has already given up.  The first probe is inline: the MMA issuer must
// not leave the tensor pipe idle while it checks a barrier that is already
// complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, ctl);
}

// Wait for a phase whose late detection costs little (a producer ahead of
// its consumers by a deep ring, a warp that waits for a whole tile): same
// contract as mbar_wait, with sleeps of at most max_ns between polls.
__device__ __forceinline__ bool mbar_wait_idle(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                               uint32_t max_ns = 256) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_idle_slow(bar, parity, ctl, max_ns);
}

// Wait used while tearing down after an abort: bounded, records nothing.
static __device__ __noinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at coordinates (x inner, y outer) into shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 2-D tiled store of a shared-memory box to global memory (rows/columns past
// the tensor's extent are not written), as part of a bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
// 3-D tiled store (the head-major output of the direct-head epilogue).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05

// Allocate `ncols` TMEM columns (power of two >= 32); whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
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

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; fp16 inputs, fp32 accumulator.
__device__ __forceinline__ void tc_mma_ts_f16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f16: fp16 A and B (both K-major), fp32 D,
// M x N tile.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                               // D format: f32
         | (0u << 7) | (0u << 10)                // A, B format: f16
         | (0u << 15) | (0u << 16)               // A, B K-major
         | ((uint32_t)(N >> 3) << 17)            // N / 8
         | ((uint32_t)(M >> 4) << 24);           // M / 16
}

// Shared-memory matrix descriptor of a K-major operand stored in the
// 128-byte swizzled layout (rows of 128 bytes, 8-row atoms of 1024 bytes).
// The tile must start on a 1024-byte boundary; advancing the start address
// by 32 bytes selects the next 16 fp16 along K inside the atom.
__device__ __forceinline__ uint64_t sdesc_sw128_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address / 16
  d |= (uint64_t)1u << 16;                   // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset: 8 rows * 128 B
  d |= (uint64_t)1u << 46;                   // descriptor version for tcgen05
  d |= (uint64_t)2u << 61;                   // swizzle: 128 B
  return d;
}

// Store 32 consecutive 32-bit TMEM columns of this thread's lane, then wait
// until the stores are complete.
__device__ __forceinline__ void tmem_st32_wait(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Store 32 consecutive 32-bit TMEM columns of this thread's lane (the
// registers are read at issue; completion is awaited with tmem_wait_st).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Store 16 consecutive 32-bit TMEM columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Wait until every tcgen05.st issued by this thread has completed.
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Load 32 consecutive 32-bit TMEM columns of this thread's lane and wait.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// ------------------------------------------------------------------ launch overlap

// Programmatic dependent launch.  The projection kernels are launched so
// that they may start while the previous kernel of the stream finishes: each
// CTA does its prologue (barriers, TMEM, descriptor prefetch), lets the next
// kernel be scheduled, and waits for the previous kernel's completion (and
// the visibility of its writes) before it touches global memory.  Launched
// without that permission, both instructions do nothing.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ clusters

// Rank of this CTA in its thread-block cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives, then waits for all:
// shared-memory writes before it are visible to peers' reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// 16-byte load from a peer CTA's shared memory (distributed shared memory).
// No memory clobber: the loads of a reduction are independent and are meant
// to be in flight together (they stay after the cluster barrier, whose
// volatile statement they follow).
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t caddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(caddr));
  return v;
}

// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace m4q
