// pkv_common.cuh -- shared device helpers of the paged-KV attention kernels
// (sm_103a): mbarrier, bulk copies, bounded waits, the sticky error word.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

// Codes recorded in the device error word (first error sticks).
enum DevErr : int32_t {
  kDevOk = 0,
  kDevBadPage = PKV_ERR_DEVICE_BOUNDS,
  kDevTimeout = PKV_ERR_DEVICE_TIMEOUT,
};

// A bounded wait gives up after this many SM clock cycles (~1 s at 2 GHz).
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ void record_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch --------------------------------------------
// A kernel launched with the programmatic stream-serialization attribute may
// begin while the kernel before it in the stream is still running.  It calls
// pdl_wait() before it reads or writes any global memory that an earlier
// kernel of the stream touches: the wait returns once those kernels have
// completed and their writes are visible.  pdl_launch_dependents() lets the
// next kernel of the stream start early (its own pdl_wait() still orders its
// memory accesses after this grid).  Both are no-ops for a plain launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after
// kWaitLimitCycles.  On give-up it records kDevTimeout and raises the CTA's
// shared abort flag; once the flag is up every later wait returns at once,
// so a kernel whose copies never land finishes in about one wait limit
// instead of one limit per wait.  Returns false when it did not see the phase.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* err,
                                                  volatile int* abort_flag,
                                                  long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      record_error(err, kDevTimeout);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// Wait for phase `parity` of `bar` whatever the abort flag says, giving up
// after `limit` cycles.  A CTA that stops early uses it to let the copies and
// tensor-core operations it has already issued land before it leaves (its
// shared memory must not be released under them).  Returns false if it gave
// up (the timeout is then recorded).
__device__ __forceinline__ bool mbar_drain_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                                long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      record_error(err, kDevTimeout);
      return false;
    }
  }
  return true;
}

// mbar_wait_bounded for a whole warp: every lane waits, and the result is
// true only if every lane saw the phase, so that the warp takes the same
// branch afterwards (lanes poll separately and may see the abort flag at
// different times).
__device__ __forceinline__ bool warp_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* err,
                                                  volatile int* abort_flag) {
  const bool ok = mbar_wait_bounded(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ---- bulk (TMA engine) copies ----------------------------------------------
// Order earlier generic-proxy shared-memory accesses before later async-proxy
// ones (a buffer is rewritten by a bulk copy after threads read it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D global -> shared bulk copy completing on `bar` (bytes % 16 == 0, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 eviction policies for streamed (read-once) and reused data.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2^x (PTX ex2.approx, flushes denormal results; 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// E4M3 pair packed in 16 bits (low byte first) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t u) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u), __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

}  // namespace pkv
