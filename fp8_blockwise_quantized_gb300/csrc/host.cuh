// Host-side helpers shared by the C-ABI translation units (api.cu, noalloc.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gmm.h"

namespace gmm {

// Records `what` and the CUDA error text for gmm_last_cuda_error() (per
// thread) and returns GMM_ERR_CUDA.
gmm_status host_cuda_fail(cudaError_t e, const char* what);
// Records a message for gmm_last_cuda_error() and returns `status`.
gmm_status host_fail(gmm_status status, const char* what);

// The bounded-wait limit handed to every kernel: GMM_WAIT_LIMIT_MS from the
// environment when set to a positive number of milliseconds (read once),
// else the built-in default.
uint64_t host_wait_limit_ns();

}  // namespace gmm
