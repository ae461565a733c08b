// Device helpers shared by the kernels of libmoe_ep: problem geometry, status bits and
// thin inline-PTX wrappers for mbarriers and 1-D TMA bulk copies (sm_90+ / sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ep.h"

namespace moe {

// Sticky device status bits: bit (1 << moe_status).
constexpr uint32_t kBitExpertRange = 1u << MOE_ERR_EXPERT_RANGE;
constexpr uint32_t kBitCapacity = 1u << MOE_ERR_CAPACITY;
constexpr uint32_t kBitRecvBound = 1u << MOE_ERR_RECV_BOUND;
constexpr uint32_t kBitTimeout = 1u << MOE_ERR_TIMEOUT;

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitBudgetNs = 2000000000ull;

// Problem geometry with the derived sizes every kernel needs.
struct Geo {
  int N, T, H, E, R, L, cap, payload;
  int64_t TR;   // pairs per rank, T*R
  int64_t RB;   // receive rows per rank, N*T*max(R,L)
  int64_t P;    // pairs in total, N*T*R
  int64_t B;    // dispatched row bytes
};

__device__ __forceinline__ void set_status(int32_t* status, uint32_t bits) {
  atomicOr(reinterpret_cast<unsigned int*>(status), bits);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch (sm_90+) ------------------------------------------
// Every kernel of the library waits for the grids it depends on before its first global
// memory access, so a kernel launched with programmatic stream serialization may be
// scheduled while its predecessor drains without changing stream-order semantics.
// Without that launch attribute both instructions are no-ops.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream launch once every CTA of this grid has called it
// (or exited). It still waits in pdl_wait() for this grid to complete.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---- mbarrier -----------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and add `bytes` to the barrier's expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of the barrier to complete, for at most kWaitBudgetNs. On expiry
// sets the timeout status bit and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitBudgetNs) {
      set_status(status, kBitTimeout);
      return false;
    }
  }
  return true;
}

// ---- 1-D TMA bulk copies ------------------------------------------------------------
// Addresses 16-byte aligned, sizes multiples of 16 bytes.

// global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global, tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src_smem)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- plain vector memory access -----------------------------------------------------

// 16-byte load that bypasses L1 (each row is read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st16(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// An L2 access policy that marks the lines it touches first to be evicted, for data a pass
// touches for the last time (PTX createpolicy, fraction 1.0).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// The opposite: lines to be kept over others, for data a later kernel of the pass reads.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ld_stream16 and st16 under an L2 access policy.
__device__ __forceinline__ uint4 ld_stream16_hint(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void st16_hint(void* p, const uint4& v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xffff0000u); }

}  // namespace moe
