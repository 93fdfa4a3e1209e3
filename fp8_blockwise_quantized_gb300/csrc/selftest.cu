// Diagnostic kernel for the failure path: a wait that nothing will ever
// complete must end in a status word, not a hang.
//
// Every wait in the library's kernels is mbar_wait: bounded by a limit on
// %globaltimer, and cut short when another role of the CTA has set the shared
// abort word.  This kernel runs exactly that code on a barrier that no thread
// and no copy ever arrives at: warp 0 waits with the caller's (short) limit,
// the other warps with a limit ten times longer, so they can only return early
// through the abort word that warp 0 sets when its own wait runs out.  The
// kernel then records the timeout bit in the workspace's sticky error word,
// exactly as the GEMM kernels do, and returns.
#include "gmm.h"
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace gmm {

__global__ void __launch_bounds__(128) wait_timeout_selftest_kernel(int32_t* ws, uint64_t limit_ns) {
  __shared__ uint64_t never;  // no arrival will ever complete its phase 0
  __shared__ volatile int abort_word;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const bool done = mbar_wait(&never, 0, &abort_word, warp == 0 ? limit_ns : 10 * limit_ns);
  __syncthreads();
  if (threadIdx.x == 0 && (!done || abort_word)) atomicOr(ws + kWsStatus, kErrTimeout);
}

}  // namespace gmm

extern "C" gmm_status gmm_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int limit_ms,
                                                void* stream) {
  if (!workspace) return GMM_ERR_WORKSPACE;
  if (workspace_bytes < 16) return GMM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return GMM_ERR_ALIGN;
  if (limit_ms < 1 || limit_ms > 10000) return GMM_ERR_SHAPE;
  gmm::wait_timeout_selftest_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int32_t*>(workspace), static_cast<uint64_t>(limit_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? GMM_OK : GMM_ERR_CUDA;
}
