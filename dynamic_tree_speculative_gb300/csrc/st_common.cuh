// Device helpers shared by the spec-tree kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_tree.h"

namespace st {

constexpr unsigned FULL = 0xffffffffu;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
// Bounded mbarrier waits: each poll may suspend the thread for up to
// WAIT_SUSPEND_NS (it wakes as soon as the phase completes); after
// WAIT_LIMIT polls (over a second) the wait gives up and reports a timeout.
constexpr uint32_t WAIT_LIMIT = 1u << 16;
constexpr uint32_t WAIT_SUSPEND_NS = 20000;

// ------------------------------------------------------------- order keys ---
// Order-preserving unsigned keys of float bit patterns: larger key <=> larger
// value, -0 and +0 equal, NaN below -inf (key 0) so that NaN never outranks a
// number, matching a stable sort that puts NaN last.

__device__ __forceinline__ bool f32_is_nan(uint32_t bits) {
  return (bits & 0x7fffffffu) > 0x7f800000u;
}

__device__ __forceinline__ uint32_t f32_key(uint32_t bits) {
  if (f32_is_nan(bits)) return 0u;
  if (bits == 0x80000000u) bits = 0u;
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

__device__ __forceinline__ uint32_t f32_from_key(uint32_t key) {
  return (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
}

// bf16: the top 16 bits of the f32 key of (bits << 16).
__device__ __forceinline__ uint32_t bf16_key(uint32_t bits16) {
  return f32_key(bits16 << 16) >> 16;
}

__device__ __forceinline__ float bf16_key_value(uint32_t key16) {
  const uint32_t bits16 = (key16 & 0x8000u) ? (key16 & 0x7fffu) : (~key16 & 0xffffu);
  return __uint_as_float(bits16 << 16);
}

// ------------------------------------------------------------- mbarriers ---

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Bounded wait on the phase with the given parity: at most `limit` polls.
// Returns false on timeout; `polls` (if given) receives the polls made.
__device__ __forceinline__ bool mbar_wait_n(uint64_t* bar, uint32_t parity, uint32_t limit,
                                            uint32_t* polls = nullptr) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity), "r"(WAIT_SUSPEND_NS)
        : "memory");
    if (done) {
      if (polls) *polls = it + 1;
      return true;
    }
  }
  if (polls) *polls = limit;
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_n(bar, parity, WAIT_LIMIT);
}

// The same with acquire at cluster scope, so that stores another CTA of the
// cluster released before its remote arrive are visible after the wait.
__device__ __forceinline__ bool mbar_wait_cluster_n(uint64_t* bar, uint32_t parity, uint32_t limit,
                                                    uint32_t* polls = nullptr) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity), "r"(WAIT_SUSPEND_NS)
        : "memory");
    if (done) {
      if (polls) *polls = it + 1;
      return true;
    }
  }
  if (polls) *polls = limit;
  return false;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  return mbar_wait_cluster_n(bar, parity, WAIT_LIMIT);
}

// L2 policy for data read again soon: evict last.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy for data read for the last time: evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Untiled bulk copy global -> shared (TMA engine), completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 16-byte read-only global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------- reductions ---

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// ------------------------------------------- programmatic dependent launch ---
// Every kernel of the library is launched with programmatic stream
// serialisation, so it may start while the previous kernel of the stream is
// finishing.  It must call grid_dependency_wait() before its first access to
// global memory that the previous kernel may touch (which makes that kernel's
// writes visible), and calls grid_dependents_launch() once the next kernel may
// begin its own launch.  Without a programmatic predecessor both are no-ops.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... Args>
cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace st
