// spec_tree_wait_selftest: runs the bounded mbarrier waits of the library's
// kernels out on purpose, on a barrier that nothing arrives on, to show that a
// wait gives up, the kernel reports SPEC_TREE_S_TIMEOUT and returns.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_tree.h"
#include "st_common.cuh"

namespace cg = cooperative_groups;

namespace st {
namespace {

// A cluster of two CTAs.  Thread 0 of each CTA sets up a barrier that expects
// one arrival and waits for its first phase with `polls` polls; nothing ever
// arrives and no copy is issued.  CTA 0 uses the CTA-scope wait of the
// support-selection kernels, CTA 1 the cluster-scope wait of the verification
// kernel.  result[2 r] = 1 if CTA r's wait gave up, result[2 r + 1] = its polls.
__global__ void __cluster_dims__(2, 1, 1) wait_selftest_kernel(uint32_t polls, uint32_t* status, uint32_t* result) {
  __shared__ uint64_t bar;
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t made = 0;
    const bool done = rank == 0 ? mbar_wait_n(&bar, 0u, polls, &made) : mbar_wait_cluster_n(&bar, 0u, polls, &made);
    result[2 * rank] = done ? 0u : 1u;
    result[2 * rank + 1] = made;
    if (!done) set_status(status, SPEC_TREE_S_TIMEOUT);
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(&bar)) : "memory");
  }
  cluster.sync();
}

}  // namespace
}  // namespace st

extern "C" int spec_tree_wait_selftest(uint32_t polls, uint32_t* status, uint32_t* result,
                                       spec_tree_stream_t stream) {
  if (status == nullptr || result == nullptr || polls == 0 || polls > st::WAIT_LIMIT) return SPEC_TREE_E_PARAM;
  st::wait_selftest_kernel<<<2, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(polls, status, result);
  return cudaGetLastError() == cudaSuccess ? SPEC_TREE_OK : SPEC_TREE_E_CUDA;
}
