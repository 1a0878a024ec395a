// mbarrier, bulk-copy (TMA) and tensor-memory PTX wrappers shared by the
// kernels, plus the bounded mbarrier wait every pipeline uses.
#pragma once

#include "common.cuh"

namespace gbf {

constexpr uint64_t kWaitBudgetNs = 1000000000ull;   // a bounded wait gives up after ~1 s ...
constexpr uint32_t kWaitMaxPolls = 1u << 23;         // ... or after this many polls (~2 s of backoff)

GBF_DEVICE uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// 32-bit shared-window accesses (addresses from smem_u32).
GBF_DEVICE uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
GBF_DEVICE float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
  return v;
}
GBF_DEVICE float lds32f(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
GBF_DEVICE void sts128f(uint32_t a, float x, float y, float z, float w) {
  asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w) : "memory");
}

GBF_DEVICE uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

GBF_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

GBF_DEVICE void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

GBF_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

GBF_DEVICE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// CLUSTER: acquire at cluster scope, for a barrier that threads of another
// CTA of the cluster arrive on (their arrive releases at cluster scope).
// HINT: the form with an explicit suspend-time hint, whose wake-up after the
// phase completes is prompter than the form without one (measured: ~5 % on
// the tcgen05 GEMM when its MMA issuer waits on TMA-filled stages this way).
constexpr uint32_t kSuspendHintNs = 64;
#define GBF_TRY_WAIT_ASM(SEM, HINTOPS)                                      \
  asm volatile("{\n\t.reg .pred p;\n\t"                                   \
               "mbarrier.try_wait.parity" SEM ".shared::cta.b64 p, [%1], %2" HINTOPS ";\n\t" \
               "selp.u32 %0, 1, 0, p;\n\t}"                                 \
               : "=r"(ok)                                                   \
               : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendHintNs)       \
               : "memory")
template <bool CLUSTER = false, bool HINT = false>
GBF_DEVICE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if (CLUSTER && HINT)
    GBF_TRY_WAIT_ASM(".acquire.cluster", ", %3");
  else if (CLUSTER)
    GBF_TRY_WAIT_ASM(".acquire.cluster", "");
  else if (HINT)
    GBF_TRY_WAIT_ASM("", ", %3");
  else
    GBF_TRY_WAIT_ASM("", "");
  return ok != 0;
}
#undef GBF_TRY_WAIT_ASM

// Bounded wait for the phase of `bar` with parity `parity` to complete.
// Gives up after kWaitBudgetNs or kWaitMaxPolls polls (whichever comes first,
// so the wait ends even if the timer were to stall), or as soon as *abort is
// set by another thread;
// a thread that gives up on its own sets *abort and the device error bit.
// SLEEP = false: no back-off between polls and the suspend-hint form of the
// poll, for the lone thread of a pipeline stage whose wake-up latency is on
// the critical path (mbarrier.try_wait itself suspends the thread until the
// phase completes or the hinted time passes, so the loop issues few
// instructions).
template <bool CLUSTER = false, bool SLEEP = true>
GBF_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, int* abort, unsigned int* err) {
  if (mbar_try_wait<CLUSTER, !SLEEP>(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  uint32_t sleep_ns = 32;
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait<CLUSTER, !SLEEP>(bar, parity)) return true;
    // back off so a waiting thread does not flood the issue slots of the
    // threads doing the work (at most ~0.25 us of extra wake-up latency)
    if (SLEEP && i > 4) {
      __nanosleep(sleep_ns);
      if (sleep_ns < 256) sleep_ns <<= 1;
    }
    if ((i & 15u) == 0) {
      if (*reinterpret_cast<volatile int*>(abort)) return false;
      if (global_timer() - t0 > kWaitBudgetNs || i >= kWaitMaxPolls) {
        raise_error(err, DEV_ERR_MBAR_TIMEOUT);
        *reinterpret_cast<volatile int*>(abort) = 1;
        return false;
      }
    }
  }
}

// mbar_wait for a whole warp with a single poller: lane 0 spins while the
// other lanes wait at the warp barrier, which issues no instructions.  (When
// every thread of a large block polls an mbarrier, the polling saturates the
// issue pipe the waits share and slows the threads doing work.)  The lanes
// observe the completed phase through lane 0's acquire and the warp barrier.
template <bool SLEEP = true>
GBF_DEVICE bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int* abort, unsigned int* err) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait<false, SLEEP>(bar, parity, abort, err) ? 1u : 0u;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// --------------------------------------------------------- bulk (1D) copies

// global -> shared, completion counted on `bar` (bytes % 16 == 0, both 16-byte aligned)
GBF_DEVICE void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// shared -> global, tracked by the issuing thread's bulk groups
GBF_DEVICE void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src_smem)),
               "r"(bytes)
               : "memory");
}

GBF_DEVICE void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// all committed bulk stores of this thread have finished reading shared memory
GBF_DEVICE void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all committed bulk stores of this thread have completed
GBF_DEVICE void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory.
GBF_DEVICE void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

}  // namespace gbf
