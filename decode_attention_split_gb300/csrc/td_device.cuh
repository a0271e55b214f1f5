// Device-side helpers shared by the td kernels: asynchronous bulk copies (TMA engine)
// into shared memory with mbarrier completion, bounded waits, and fp32 widening of
// stored elements.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "td.h"

namespace td {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// A wait on an asynchronous copy gives up after this many SM cycles (about one second)
// and reports TD_DEV_WAIT_TIMEOUT instead of hanging the GPU.
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later
// asynchronous-proxy accesses (a bulk copy overwriting a buffer just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One arrival (release semantics at CTA scope: this thread's earlier accesses happen before
// the phase completes for a waiter).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Waits for phase `parity` of an mbarrier to complete; false once `limit` SM cycles have
// passed without it.
__device__ __forceinline__ bool mbar_wait_bounded_for(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// The kernels' wait: false after kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  return mbar_wait_bounded_for(bar, parity, kWaitLimitCycles);
}

// Orders this thread's earlier generic-proxy global accesses (and those it has observed, e.g.
// partials other CTAs published before an atomic ticket) before its later asynchronous-proxy
// (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Programmatic dependent launch: wait until the grids this one depends on have completed and
// their writes are visible; allow the next grid in the stream to be scheduled early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 policy for data read exactly once (the KV stream): evict it first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Warms L2 with `bytes` (a multiple of 16) from a 16-byte aligned global address. A hint:
// nothing waits for it.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// A load that may race with another grid's store to the same word (the value is only used
// as a guess).
__device__ __forceinline__ int32_t ld_relaxed(const int32_t *p) {
  int32_t v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// A load with acquire semantics at GPU scope (a completion counter other CTAs release to).
__device__ __forceinline__ int32_t ld_acquire(const int32_t *p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One bulk copy global -> shared through the TMA engine; completion is counted on `bar`
// in bytes. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Bulk copy global -> shared without a cache hint (16-byte multiples, as bulk_g2s).
__device__ __forceinline__ void bulk_g2s_plain(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Ticket on a completion counter: release (the CTA's partial writes, ordered before this by
// a barrier, become visible first) and acquire (other CTAs' released writes are visible
// after it). Returns the previous count.
__device__ __forceinline__ int ticket_acq_rel(int *cnt) {
  int prev;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(cnt) : "memory");
  return prev;
}

// ---- thread-block clusters ---------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster: writes before it (shared or global) are visible
// to the cluster after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Generic address of the variable at `p` (this CTA's shared memory) in CTA `rank`.
template <typename T>
__device__ __forceinline__ const T *map_to_rank(const T *p, uint32_t rank) {
  uint64_t out;
  asm volatile("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(p), "r"(rank));
  return reinterpret_cast<const T *>(out);
}

// ---- widening of stored elements to fp32 ----------------------------------------------

__device__ __forceinline__ float widen_elem(float x) { return x; }
__device__ __forceinline__ float widen_elem(__nv_bfloat16 x) { return __bfloat162float(x); }

// A bf16 value is the upper half of a binary32 value.
__device__ __forceinline__ void widen_bf16x2(uint32_t w, float &lo, float &hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

// Loads N consecutive elements of type E from shared or global memory at p (aligned to
// N * sizeof(E) bytes, which is 4, 8 or 16) and widens them to fp32.
template <typename E, int N>
__device__ __forceinline__ void load_widen(const void *p, float (&f)[N]) {
  if constexpr (sizeof(E) == 4) {
    static_assert(N == 2 || N == 4, "fp32 vector of 2 or 4");
    if constexpr (N == 4) {
      const float4 x = *reinterpret_cast<const float4 *>(p);
      f[0] = x.x, f[1] = x.y, f[2] = x.z, f[3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2 *>(p);
      f[0] = x.x, f[1] = x.y;
    }
  } else {
    static_assert(N == 2 || N == 4 || N == 8, "bf16 vector of 2, 4 or 8");
    if constexpr (N == 8) {
      const uint4 x = *reinterpret_cast<const uint4 *>(p);
      widen_bf16x2(x.x, f[0], f[1]);
      widen_bf16x2(x.y, f[2], f[3]);
      widen_bf16x2(x.z, f[4], f[5]);
      widen_bf16x2(x.w, f[6], f[7]);
    } else if constexpr (N == 4) {
      const uint2 x = *reinterpret_cast<const uint2 *>(p);
      widen_bf16x2(x.x, f[0], f[1]);
      widen_bf16x2(x.y, f[2], f[3]);
    } else {
      const uint32_t x = *reinterpret_cast<const uint32_t *>(p);
      widen_bf16x2(x, f[0], f[1]);
    }
  }
}

template <typename E>
__device__ __forceinline__ void store_elem(E *p, float x);
template <>
__device__ __forceinline__ void store_elem<float>(float *p, float x) {
  *p = x;
}
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16 *p, float x) {
  *p = __float2bfloat16_rn(x);
}

__device__ __forceinline__ void report(uint32_t *status, uint32_t bits) {
  if (status != nullptr && bits != 0u) atomicOr(status, bits);
}

}  // namespace td
