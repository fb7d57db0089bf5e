// Device-side helpers shared by the FusedKV kernels: mbarriers, bulk (TMA)
// copies, bounded waits and the device status word.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fkv_kernels.h"

namespace fkv {

// Bits of the device status word (one int32 per context).
enum : int {
  kDevOk = 0,
  kDevBadArg = 1,    // a sequence length / append position out of range
  kDevTimeout = 2,   // a bounded wait ran out
};

// kWaitLimitNs (fkv_kernels.h) is the default wall-clock limit of every spin
// on an mbarrier.  Nothing legitimate waits that long; a wait that runs out
// sets kDevTimeout and the kernel returns.  Draining copies already in flight
// after such a timeout has its own limit:
constexpr unsigned long long kDrainLimitNs = 50000000ull;   // 50 ms

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream is still
// running.  grid_dep_wait() blocks until the predecessor grid has completed and
// its memory is visible, so every kernel calls it before its first global
// memory access; grid_dep_trigger() lets the successor be scheduled early.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void flag_status(int* status, int bit) {
  if (status) atomicOr(status, bit);
}

// The limit of the bounded waits of one launch.  Each context keeps it in a
// device word beside its status word (kWaitLimitNs unless a test lowered it),
// so that a launch replayed from a CUDA graph reads the current setting.
// Read after grid_dep_wait().
__device__ __forceinline__ unsigned long long wait_limit_ns(const unsigned long long* word) {
  return word ? *word : kWaitLimitNs;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order earlier generic-proxy shared-memory accesses before later async-proxy
// (TMA) accesses of the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

// Spin until the phase with the given parity completes, or until `limit_ns`
// of wall-clock time has passed.  Returns false on timeout.  A limit of 0
// reports a timeout at once, without looking at the barrier: the failure
// path's test setting (see wait_limit_ns above), which takes every kernel
// down its timeout path at its first wait, whatever the timing.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Bulk (non-tensor) asynchronous copy global -> shared, completing `bytes`
// transactions on `bar`.  dst and src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// An L2 policy that marks streamed cache tiles evict-first: each KV byte is
// read once per call.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// bf16 pair in a 32-bit word -> two fp32 (exact: bf16 is the top half of fp32).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& w, float* f);

template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& w, float* f) {
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
  f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
  f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

template <>
__device__ __forceinline__ void unpack16<float>(const uint4& w, float* f) {
  f[0] = __uint_as_float(w.x);
  f[1] = __uint_as_float(w.y);
  f[2] = __uint_as_float(w.z);
  f[3] = __uint_as_float(w.w);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace fkv
