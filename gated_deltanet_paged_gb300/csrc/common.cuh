// common.cuh -- device and host helpers shared by the GDN kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA tensor loads and the tcgen05 tensor
// core (TMEM allocation, MMA issue / commit, TMEM loads), plus the host-side
// status plumbing of the C ABI.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_paged.h"

namespace gdn {

constexpr int kDimK = 128;  // key dimension K
constexpr int kDimV = 128;  // value dimension V
constexpr int kChunk = 64;  // tokens per chunk

// ---------------------------------------------------------------------------
// Device-side error reporting: kernels record the first violation they see in
// the caller's err_word (when one is given) as (kind << 24) | sequence.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_error(int32_t* err_word, int kind, int seq) {
  if (err_word) atomicCAS(err_word, 0, (kind << 24) | (seq & 0xFFFFFF));
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As above, but the thread may be suspended in the instruction for up to
// ~1 ms while the phase is incomplete (no busy polling).
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Non-blocking test of phase `parity`.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after limit_ns (~2 s by
// default).  Returns false on time-out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// As mbar_wait, but also gives up as soon as *abort becomes non-zero (another
// thread of the CTA timed out).
// The thread sleeps in the wait instruction (no issue slots taken from the
// warps that work) until the phase completes or ~1 ms passes.  The loop is a
// function of its own, so that the many call sites in a kernel's hot loop each
// carry only the first test.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > 2000000000ull) return false;
  }
}
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort);
}

// Proxy fence: makes this thread's generic-proxy shared-memory writes visible
// to the async proxy (tensor core, TMA) after the next barrier.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA: 3-D tiled tensor load into shared memory, completing on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// 2-D tiled tensor load (coordinates: inner, outer).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// 3-D tiled tensor store from shared memory (bulk group of this thread);
// rows outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int32_t c0, int32_t c1,
                                             int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// 2-D tiled tensor store from shared memory (bulk group of this thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until this thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Programmatic dependent launch.  Kernels launched with programmatic stream
// serialisation (gdn_host::launch_pdl) may start while the kernel before them on
// the stream finishes; pdl_wait blocks until that kernel has completed and its
// memory is visible (it returns at once for a plain launch), and
// pdl_launch_dependents lets the next kernel on the stream begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor core.
// ---------------------------------------------------------------------------
// Allocate `ncols` TMEM columns (power of two >= 32); the whole warp executes
// it and the base address lands in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (fp16 or bf16 operands, fp32 accumulate).
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four (two) consecutive K-steps of one product, issued as a single asm block:
// step s uses descriptors a + s*astep and b + s*bstep (steps in 16-byte units
// of the start-address field); the first step accumulates iff acc0 != 0, the
// others always accumulate.
__device__ __forceinline__ void tc_mma4(uint32_t d, uint64_t a, uint32_t astep, uint64_t b, uint32_t bstep,
                                        uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 q, %6, %6;\n\t"
      "add.s64 a1, %1, %2;\n\tadd.s64 a2, a1, %2;\n\tadd.s64 a3, a2, %2;\n\t"
      "add.s64 b1, %3, %4;\n\tadd.s64 b2, b1, %4;\n\tadd.s64 b3, b2, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %3, %5, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %5, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %5, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %5, q;\n\t}\n" ::"r"(d),
      "l"(a), "l"(static_cast<uint64_t>(astep)), "l"(b), "l"(static_cast<uint64_t>(bstep)), "r"(idesc), "r"(acc0)
      : "memory");
}
__device__ __forceinline__ void tc_mma2(uint32_t d, uint64_t a, uint32_t astep, uint64_t b, uint32_t bstep,
                                        uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, b1;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 q, %6, %6;\n\t"
      "add.s64 a1, %1, %2;\n\tadd.s64 b1, %3, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %3, %5, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %5, q;\n\t}\n" ::"r"(d),
      "l"(a), "l"(static_cast<uint64_t>(astep)), "l"(b), "l"(static_cast<uint64_t>(bstep)), "r"(idesc), "r"(acc0)
      : "memory");
}

// Same with the A operand in TMEM (lane m = row m, column c = elements 2c and
// 2c+1 of the K dimension, fp16/bf16 pairs); astep in TMEM columns.
__device__ __forceinline__ void tc_mma4_ts(uint32_t d, uint32_t a_tmem, uint32_t astep, uint64_t b, uint32_t bstep,
                                           uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 q, %6, %6;\n\t"
      "add.u32 a1, %1, %2;\n\tadd.u32 a2, a1, %2;\n\tadd.u32 a3, a2, %2;\n\t"
      "add.s64 b1, %3, %4;\n\tadd.s64 b2, b1, %4;\n\tadd.s64 b3, b2, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %3, %5, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %5, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %5, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %5, q;\n\t}\n" ::"r"(d),
      "r"(a_tmem), "r"(astep), "l"(b), "l"(static_cast<uint64_t>(bstep)), "r"(idesc), "r"(acc0)
      : "memory");
}
__device__ __forceinline__ void tc_mma2_ts(uint32_t d, uint32_t a_tmem, uint32_t astep, uint64_t b, uint32_t bstep,
                                           uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 a1;\n\t.reg .b64 b1;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 q, %6, %6;\n\t"
      "add.u32 a1, %1, %2;\n\tadd.s64 b1, %3, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %3, %5, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %5, q;\n\t}\n" ::"r"(d),
      "r"(a_tmem), "r"(astep), "l"(b), "l"(static_cast<uint64_t>(bstep)), "r"(idesc), "r"(acc0)
      : "memory");
}

// Store 16 (8) consecutive 32-bit columns of this thread's TMEM lane and wait.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// The same stores and fragment loads without their wait (several in flight;
// tmem_wait_st / tmem_wait_ld before the values are used or published).
__device__ __forceinline__ void tmem_st16_nw(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld16x256_x4_nw(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// Wait for two fragment loads in flight; the registers are operands so that no
// use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld2(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                 "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}

// Load 32 consecutive fp32 columns of this thread's TMEM lane and wait for them.
// 16 lanes x 32 columns, twice: threads 0-15 read lanes 0-15 of the warp's
// quarter at columns [col, col + 32), threads 16-31 the same lanes at columns
// [col + 32, col + 64) -- the rows of an M = 64 accumulator (its row m sits in
// lane 32 (m / 16) + m % 16).
__device__ __forceinline__ void tmem_ld16x32bx2_32(uint32_t taddr, float (&r)[32]) {
  uint32_t* u = reinterpret_cast<uint32_t*>(r);
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32], 32;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
        "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]),
        "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]),
        "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]),
        "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
  uint32_t* u = reinterpret_cast<uint32_t*>(r);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
        "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]),
        "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]),
        "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]),
        "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
      : "r"(taddr)
      : "memory");
}

// Load a 16-lane x 32-column fp32 block (four 16 x 8 repeats) in the fragment
// layout of the 16x256b shape, and wait for it: in repeat j, thread i holds
// columns 8 j + 2 (i % 4) and + 1 of lane i / 4 (r[4 j], r[4 j + 1]) and of lane
// i / 4 + 8 (r[4 j + 2], r[4 j + 3]).  taddr's lane is the first of the 16.
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Four 8 x 8 b16 matrices in the fragment layout above (thread i: row i / 4,
// elements 2 (i % 4) and + 1 of each) stored transposed: row k of matrix m
// (column k of the fragment) goes to the 16 bytes at thread 8 m + k's address.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, uint32_t m0, uint32_t m1, uint32_t m2,
                                                  uint32_t m3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(m0),
               "r"(m1), "r"(m2), "r"(m3)
               : "memory");
}

// Load 64 consecutive fp32 columns of this thread's TMEM lane and wait for them.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&r)[64]) {
  uint32_t* u = reinterpret_cast<uint32_t*>(r);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31]), "=r"(u[32]), "=r"(u[33]), "=r"(u[34]), "=r"(u[35]), "=r"(u[36]), "=r"(u[37]), "=r"(u[38]), "=r"(u[39]), "=r"(u[40]), "=r"(u[41]), "=r"(u[42]), "=r"(u[43]), "=r"(u[44]), "=r"(u[45]), "=r"(u[46]), "=r"(u[47]), "=r"(u[48]), "=r"(u[49]), "=r"(u[50]), "=r"(u[51]), "=r"(u[52]), "=r"(u[53]), "=r"(u[54]), "=r"(u[55]), "=r"(u[56]), "=r"(u[57]), "=r"(u[58]), "=r"(u[59]), "=r"(u[60]), "=r"(u[61]), "=r"(u[62]), "=r"(u[63])
      : "r"(taddr)
      : "memory");
}

// Load 16 consecutive fp32 columns of this thread's TMEM lane and wait for them.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
  uint32_t* u = reinterpret_cast<uint32_t*>(r);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
        "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]),
        "=r"(u[15])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B: 8 rows of 128 B per 1024 B atom, 16-byte
// chunk c of row r stored at chunk c ^ (r % 8)).  lbo / sbo in bytes.
//   K-major operand: rows (M or N) 128 B apart, sbo = stride between 8-row
//     groups; a K step of 16 elements inside the atom advances the start by 32 B.
//   MN-major operand: 128 B rows hold 64 consecutive M/N elements of one k;
//     sbo = stride between 8-k groups, lbo = stride between 64-element M/N blocks.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16 with an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_bf16, bool b_bf16, bool a_mn_major,
                                                 bool b_mn_major) {
  return (1u << 4) | ((a_bf16 ? 1u : 0u) << 7) | ((b_bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of 16-byte chunk `c` of row `r` in a 128B-swizzled tile.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_half2(float2 x) { return pack_half2(x.x, x.y); }
__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf162(float2 x) { return pack_bf162(x.x, x.y); }
__device__ __forceinline__ float2 unpack_bf162(uint32_t u) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(h);
}

}  // namespace gdn

// ---------------------------------------------------------------------------
// Host-side helpers of the C ABI.
// ---------------------------------------------------------------------------
namespace gdn_host {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// GDN_OK if the current device is an sm_103 part, else GDN_ERR_UNSUPPORTED
// (or GDN_ERR_CUDA when no device can be queried).
int check_device(int* sm_count);

// Encode a 3-D bf16 tensor map over [T, H, D] (D innermost) with a box of
// 64 elements x 1 head x 64 tokens and 128-byte swizzle.
int encode_tokens_map(CUtensorMap* map, const void* base, int64_t T, int64_t H, int64_t D);

// Encode a 2-D fp16 tensor map over [rows, cols] (cols a multiple of 64) with
// a box of 64 x 64 and 128-byte swizzle.
int encode_tiles_map_f16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols);
int encode_tokens_map_32(CUtensorMap* map, const void* base, int64_t T, int64_t H, int64_t D);  // 64B swizzle

inline int launch_status() { return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// cudaFuncSetAttribute once per device (the setting lasts for the process):
// `done` is the call site's mask of devices already set.
template <typename... Params>
inline int func_attr_once(void (*kernel)(Params...), cudaFuncAttribute attr, int value, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return GDN_OK;
  if (cudaFuncSetAttribute(kernel, attr, value) != cudaSuccess) {
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return GDN_OK;
}

// Launch as a programmatic dependent of the previous kernel on the stream (the
// kernel calls pdl_wait before it reads anything that kernel may write).
template <typename... Params, typename... Args>
inline int launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn_host
