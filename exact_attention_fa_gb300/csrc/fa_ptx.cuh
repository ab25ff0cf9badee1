// Inline-PTX building blocks for the sm_103a kernels: mbarriers with bounded waits, TMA tile
// loads, tcgen05 (TMEM allocation, MMA, commit, TMEM loads/stores) and the shared-memory /
// instruction descriptors the tensor cores read.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace fa {

// ------------------------------------------------------------------------------------------
// error reporting from device code
// ------------------------------------------------------------------------------------------
// Bits of the device error word (the host reads and clears it through fa_check_device_error).
enum : unsigned {
  kErrTimeout = 1u,      // a bounded wait (mbarrier or counter) gave up
  kErrSmemAlign = 2u,    // dynamic shared memory not 1024-byte aligned
};

// Per-CTA control block in shared memory: an abort flag that every bounded wait polls, so that
// when one warp gives up the others stop waiting too.
struct Ctl {
  volatile int* abort_flag;
  unsigned* err;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void raise_error(const Ctl& c, unsigned bits) {
  atomicOr(c.err, bits);
  *c.abort_flag = 1;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Producer-side barrier arrive and TMA issue are executed by the whole (converged) producer warp;
// one elected lane performs them, as for the MMA helpers below.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the thread sleep in hardware (up to `ns`) until the phase completes, so that
// waiting warps do not take issue slots from the working warps of their SM sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity of the barrier has completed. Bounded: gives up
// (returning false, raising kErrTimeout and the CTA abort flag) after ctl.timeout_ns of wall
// time, or as soon as another warp of the CTA has aborted.
// After the first failed test, waiting threads sleep in hardware (up to this many ns per try,
// woken early when the phase completes) instead of spinning; 0 disables the sleep.
#ifndef FA_WAIT_SLEEP_NS
#define FA_WAIT_SLEEP_NS 200000
#endif
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (FA_WAIT_SLEEP_NS ? mbar_try_wait_sleep(bar, parity, FA_WAIT_SLEEP_NS)
                         : mbar_try_wait(bar, parity))
      return true;
    if (*ctl.abort_flag) return false;
    if (globaltimer() - t0 > ctl.timeout_ns) {
      raise_error(ctl, kErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same bounded wait by polling, never suspending: for the single thread that issues MMAs, which
// must resume within a few cycles of the phase completing to keep the tensor pipe fed (a thread
// suspended in try_wait takes a few hundred cycles to resume).
__device__ __forceinline__ bool mbar_wait_poll(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  if (mbar_test_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (*ctl.abort_flag) return false;
      if (globaltimer() - t0 > ctl.timeout_ns) {
        raise_error(ctl, kErrTimeout);
        return false;
      }
    }
  }
}

// Waits of the converged MMA-issuing warp: every lane waits and all lanes take the same outcome.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl));
}
__device__ __forceinline__ bool mbar_wait_poll_warp(uint32_t bar, uint32_t parity, const Ctl& ctl) {
  return __all_sync(0xffffffffu, mbar_wait_poll(bar, parity, ctl));
}

// Per-warpgroup register budgets (executed by all warps of a warpgroup): a warpgroup that needs
// few registers gives them back, one that needs many takes them. The sum over the CTA's
// warpgroups must stay within what the launch allocated.
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion counted in bytes on an mbarrier)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e prefetch.tensormap [%0];\n\t}" ::"l"(map)
      : "memory");
}
// Contiguous global -> shared copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// completing on mbarrier `bar`. Whole warp; one elected lane issues.
__device__ __forceinline__ void tma_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      "\n\t}" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n\t}" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Bulk tensor reduction shared -> global: adds a swizzled fp32 shared-memory box into the tensor
// (element-wise, performed at L2), tracked by the issuing thread's bulk async-group.
// Tensor store shared -> global of one box (issued by a single thread; rows past the tensor's
// extent are not written).
__device__ __forceinline__ void tma_store_3d(const void* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          map),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_reduce_add_3d(const void* map, uint32_t src, int c0, int c1,
                                                  int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(map),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until the shared memory of every committed bulk operation has been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk operation has completed (its global writes are done).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Named barrier over `count` threads that also ORs a predicate across them: every participant
// gets the same answer, so a group can leave a loop together (never stranding a barrier).
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.b32 pin, %1, 0;\n\t"
      "bar.red.or.pred pout, %2, %3, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}\n"
      : "=r"(out)
      : "r"(v ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Makes generic-proxy shared-memory writes of this thread visible to the async proxy (TMA,
// tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bounded wait until the 32-bit counter at ctr reaches at least want (the counter only grows
// while the wait lasts). Polls with acquire loads at gpu scope; gives up like mbar_wait.
__device__ __forceinline__ bool wait_counter_geq(const unsigned* ctr, unsigned want,
                                                 const Ctl& ctl) {
  auto load = [&]() {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    return v;
  };
  if (load() >= want) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    __nanosleep(256);
    if (load() >= want) return true;
    if (*ctl.abort_flag) return false;
    if (globaltimer() - t0 > ctl.timeout_ns) {
      raise_error(ctl, kErrTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit
// ------------------------------------------------------------------------------------------
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

// MMA and commit helpers are executed by a whole converged warp: each asm block elects one lane
// (elect.sync, the same lane every time) to issue the tcgen05 instructions. Issued this way the
// descriptors stay warp-uniform; issuing from a one-lane branch instead was measured ~3x slower
// per MMA when busy warps share the SM sub-partition.
//
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate. `accumulate` = 0 overwrites D.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives (once) on the mbarrier when every tcgen05 operation issued so far by the elected lane
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Tensor-memory loads/stores, 32x32b shape: thread t of the warp reads/writes lane
// (32*(warp%4) + t) and N consecutive 32-bit columns. The load waits for completion inside the
// same asm statement so that the compiler cannot consume the registers early.
#define FA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                 "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define FA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                 "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr)
      : "memory");
}
// 128 consecutive columns in one load and one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
      "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
      "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
      "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
      "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, "
      "[%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24), FA_R8(32), FA_R8(40), FA_R8(48), FA_R8(56),
        FA_R8(64), FA_R8(72), FA_R8(80), FA_R8(88), FA_R8(96), FA_R8(104), FA_R8(112), FA_R8(120)
      : "r"(taddr)
      : "memory");
}
// 128 consecutive columns as two 64-column loads and one wait: the same result as tmem_ld128,
// but no single instruction needs 128 destination registers, so it also compiles where the
// register budget is raised per warpgroup.
__device__ __forceinline__ void tmem_ld64x2(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63"
      "}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
      "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
      "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
      "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127"
      "}, [%129];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24), FA_R8(32), FA_R8(40), FA_R8(48), FA_R8(56),
        FA_R8(64), FA_R8(72), FA_R8(80), FA_R8(88), FA_R8(96), FA_R8(104), FA_R8(112), FA_R8(120)
      : "r"(taddr), "r"(taddr + 64u)
      : "memory");
}
// 16 consecutive columns in one load and one wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8)
      : "r"(taddr)
      : "memory");
}
// 64 consecutive columns in one load and one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63"
      "}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24), FA_R8(32), FA_R8(40), FA_R8(48), FA_R8(56)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      FA_W8(0), FA_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                   taddr),
               FA_W8(0)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
#undef FA_R8
#undef FA_W8

// ------------------------------------------------------------------------------------------
// shared-memory matrix descriptors (start, leading- and stride-dimension byte offsets in 16-byte
// units at bits 0-13, 16-29, 32-45; version 1 at bit 46; layout type at bits 61-63)
// ------------------------------------------------------------------------------------------
// Descriptor of an operand without swizzle, K-major, in 8-row x 16-byte core matrices (128
// contiguous bytes each): lbo = byte distance between the core matrices of one 8-row group that
// are adjacent along K, sbo = byte distance between adjacent 8-row groups. Layout type 0.
__device__ __forceinline__ uint64_t sdesc_none(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  return d;
}

// A 128-byte-swizzled operand (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B), as two
// 32-bit halves so that the MMA issue loop only adds a constant to the low half per K-step.
//   K-major tile (rows of 64 bf16 = 128 B): SBO = 1024 (next group of 8 rows); LBO unused.
//   MN-major tile: LBO = byte distance to the next 64-element block along M/N, SBO = 1024 (next
//   group of 8 rows along K). Layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_hi_sw128(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}

// Lean issue of a whole 128 x 128 (x K) product for the MMA warp, which shares its SM
// sub-partition with busy warps: every MMA is one 64-bit add and the tcgen05.mma itself.
// a[k]: precomputed A descriptors per K-step; b: B descriptor of step 0, K-major 128-byte swizzle
// with 64-column boxes 16 KB apart (steps at +0, +2, +4, +6 then +1024.. in 16-byte units).
__device__ __forceinline__ void mma_qk_d128(uint32_t d_tmem, const uint64_t (&a)[8], uint64_t b,
                                            uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .b64 tb;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %10, 0;\n\t"
      "add.s64 tb, %9, 2;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, tb, %10, 1;\n\t"
      "add.s64 tb, %9, 4;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, tb, %10, 1;\n\t"
      "add.s64 tb, %9, 6;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, tb, %10, 1;\n\t"
      "add.s64 tb, %9, 1024;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, tb, %10, 1;\n\t"
      "add.s64 tb, %9, 1026;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, tb, %10, 1;\n\t"
      "add.s64 tb, %9, 1028;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, tb, %10, 1;\n\t"
      "add.s64 tb, %9, 1030;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, tb, %10, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]),
      "l"(b), "r"(idesc)
      : "memory");
}
__device__ __forceinline__ void mma_qk_d64(uint32_t d_tmem, const uint64_t (&a)[4], uint64_t b,
                                           uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .b64 tb;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %6, 0;\n\t"
      "add.s64 tb, %5, 2;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, tb, %6, 1;\n\t"
      "add.s64 tb, %5, 4;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, tb, %6, 1;\n\t"
      "add.s64 tb, %5, 6;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, tb, %6, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b), "r"(idesc)
      : "memory");
}
// Eight K-steps of a product with both operands in shared memory, each step's descriptors given
// (a[k], b[k]); the first step overwrites D unless accumulate is set.
__device__ __forceinline__ void mma_ss_k8(uint32_t d_tmem, const uint64_t (&a)[8],
                                          const uint64_t (&b)[8], uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %18, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %17, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %17, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %17, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %17, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %17, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %17, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %17, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %17, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]),
      "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
      "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same over four K-steps, overwriting D.
__device__ __forceinline__ void mma_ss_k4(uint32_t d_tmem, const uint64_t (&a)[8],
                                          const uint64_t (&b)[8], uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %9, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %9, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %9, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %9, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
      "r"(idesc)
      : "memory");
}
// O (+)= P V over 128 keys: A = P in TMEM (8 columns per K-step), B = V MN-major (16 rows = 2 KB
// per K-step, i.e. +128 in 16-byte units).
__device__ __forceinline__ void mma_pv_k128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .pred p;\n\t.reg .b64 tb;\n\t.reg .b32 ta;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.s32 ta, %1, 8;\n\tadd.s64 tb, %2, 128;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 16;\n\tadd.s64 tb, %2, 256;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 24;\n\tadd.s64 tb, %2, 384;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 32;\n\tadd.s64 tb, %2, 512;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 40;\n\tadd.s64 tb, %2, 640;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 48;\n\tadd.s64 tb, %2, 768;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 56;\n\tadd.s64 tb, %2, 896;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (+)= A B over K = 128 with A read from TMEM at 8-column groups {0, 8, 16, 24, 64, 72, 80, 88}
// (two 64-column halves, each packed into its first 32 columns) and B MN-major in shared memory
// (+2 KB per K-step). `accumulate` applies to the first step; the rest accumulate.
__device__ __forceinline__ void mma_ts_k128_halves(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .pred p;\n\t.reg .b64 tb;\n\t.reg .b32 ta;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.s32 ta, %1, 8;\n\tadd.s64 tb, %2, 128;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 16;\n\tadd.s64 tb, %2, 256;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 24;\n\tadd.s64 tb, %2, 384;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 64;\n\tadd.s64 tb, %2, 512;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 72;\n\tadd.s64 tb, %2, 640;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 80;\n\tadd.s64 tb, %2, 768;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 88;\n\tadd.s64 tb, %2, 896;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D = A B over K = 128 with both operands MN-major in shared memory (+2 KB per K-step each).
__device__ __forceinline__ void mma_ss_k128_mn(uint32_t d_tmem, uint64_t a, uint64_t b,
                                               uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .b64 ta, tb;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 0;\n\t"
      "add.s64 ta, %1, 128;\n\tadd.s64 tb, %2, 128;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ta, tb, %3, 1;\n\t"
      "add.s64 ta, %1, 256;\n\tadd.s64 tb, %2, 256;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ta, tb, %3, 1;\n\t"
      "add.s64 ta, %1, 384;\n\tadd.s64 tb, %2, 384;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ta, tb, %3, 1;\n\t"
      "add.s64 ta, %1, 512;\n\tadd.s64 tb, %2, 512;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ta, tb, %3, 1;\n\t"
      "add.s64 ta, %1, 640;\n\tadd.s64 tb, %2, 640;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ta, tb, %3, 1;\n\t"
      "add.s64 ta, %1, 768;\n\tadd.s64 tb, %2, 768;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ta, tb, %3, 1;\n\t"
      "add.s64 ta, %1, 896;\n\tadd.s64 tb, %2, 896;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], ta, tb, %3, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc)
      : "memory");
}
// 8-bit operands (tcgen05.mma kind::f8f6f4, e4m3 A and B, fp32 accumulate): one K-step is 32
// elements = 32 bytes, the same byte width as a 16-bit K-step, so a K-major 128-byte-swizzled
// tile (rows of 128 e4m3) advances its descriptor by 2 (16-byte units) per step.
// S = Q K^T at d = 128: four K-steps inside one swizzle atom row, A and B both K-major.
__device__ __forceinline__ void mma_qk_f8_d128(uint32_t d_tmem, const uint64_t (&a)[4], uint64_t b,
                                               uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .b64 tb;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %5, %6, 0;\n\t"
      "add.s64 tb, %5, 2;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %2, tb, %6, 1;\n\t"
      "add.s64 tb, %5, 4;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, tb, %6, 1;\n\t"
      "add.s64 tb, %5, 6;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %4, tb, %6, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b), "r"(idesc)
      : "memory");
}
// O (+)= P V over 128 keys with e4m3 operands: A = P in TMEM (four e4m3 per 32-bit column, so a
// 32-key K-step is 8 columns), B = V MN-major (rows of 128 e4m3; 32 keys = four 8-row groups =
// 4 KB per K-step, i.e. +256 in 16-byte units).
__device__ __forceinline__ void mma_pv_f8_k128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .pred p;\n\t.reg .b64 tb;\n\t.reg .b32 ta;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t"
      "add.s32 ta, %1, 8;\n\tadd.s64 tb, %2, 256;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 16;\n\tadd.s64 tb, %2, 512;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], tb, %3, 1;\n\t"
      "add.s32 ta, %1, 24;\n\tadd.s64 tb, %2, 768;\n\t@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ta], tb, %3, 1;\n\t"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__host__ __device__ constexpr uint64_t sdesc64(uint32_t lo, uint32_t hi) {
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 D, dense.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   15 A major (0 = K, 1 = MN), 16 B major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn_major) << 15) |
         (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with e4m3 A and B (format code 0 in bits
// 7-9 and 10-12), fp32 D, dense; the other fields as in idesc_bf16.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(a_mn_major) << 15) |
         (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------------------------------
// small math helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed pairs of fp32 (Blackwell's two-wide FP32 datapath): one instruction for two values.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// 2^x for two values on the FMA pipes instead of the SFU (the FA4 idea of "3 · FlashAttention",
// 3.5: a share of the exponentials computed in software). x = j + f with j = rint(x), f in
// [-1/2, 1/2]: adding 1.5 * 2^23 leaves j in the low mantissa bits; 2^f comes from a degree-3
// polynomial fitted to 2^f in relative error on [-1/2, 1/2] by the Remez exchange algorithm
// (coefficients from exact_attention_fa_gb300/exp2_poly_fit.py, max relative error 7.5e-5 in fp32,
// far below the bf16 rounding of P); j is then added into the exponent field. x below -126
// (masked keys, -inf) gives exactly 0, as the SFU's flush-to-zero ex2 does.
constexpr float kExp2C0 = 0.9999280571937561f;
constexpr float kExp2C1 = 0.6932609677314758f;
constexpr float kExp2C2 = 0.2426111251115799f;
constexpr float kExp2C3 = 0.0551716685295105f;
__device__ __forceinline__ void exp2_poly2(float x0, float x1, float& p0, float& p1) {
  constexpr float kRound = 12582912.f;  // 1.5 * 2^23
  const unsigned long long x = f2_pack(fmaxf(x0, -127.f), fmaxf(x1, -127.f));
  const unsigned long long t = f2_add(x, f2_pack(kRound, kRound));
  const unsigned long long jf = f2_add(t, f2_pack(-kRound, -kRound));  // rint(x) as a float
  const unsigned long long f = f2_fma(jf, f2_pack(-1.f, -1.f), x);      // x - rint(x)
  unsigned long long q = f2_fma(f2_pack(kExp2C3, kExp2C3), f, f2_pack(kExp2C2, kExp2C2));
  q = f2_fma(q, f, f2_pack(kExp2C1, kExp2C1));
  q = f2_fma(q, f, f2_pack(kExp2C0, kExp2C0));
  float t0, t1, q0, q1;
  f2_unpack(t, t0, t1);
  f2_unpack(q, q0, q1);
  const int j0 = static_cast<int>(__float_as_uint(t0)) - static_cast<int>(__float_as_uint(kRound));
  const int j1 = static_cast<int>(__float_as_uint(t1)) - static_cast<int>(__float_as_uint(kRound));
  p0 = x0 < -126.f ? 0.f : __int_as_float(__float_as_int(q0) + (j0 << 23));
  p1 = x1 < -126.f ? 0.f : __int_as_float(__float_as_int(q1) + (j1 << 23));
}

// Four fp32 values rounded to e4m3 (nearest, ties to even, saturating at +-448), packed with the
// first in the lowest byte. cvt's first source goes to the upper byte of each pair.
__device__ __forceinline__ uint32_t pack_e4m3x4(float p0, float p1, float p2, float p3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(p0), "f"(p1), "f"(p2), "f"(p3));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace fa
