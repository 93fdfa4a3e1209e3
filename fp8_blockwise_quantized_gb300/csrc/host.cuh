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

// The FP8 forward's kernel when the tile configuration leaves cta_group 0
// (one CTA per tile for every shape).
int host_fp8_default_cta_group(int64_t N, int fuse, int bn, int ctas);
// Resolves an FP8 tile configuration (NULL or 0 fields: the defaults) into
// *out with every field set; GMM_ERR_UNSUPPORTED for a value outside the set
// gmm.h documents.  sms = 0 checks only the rules that do not depend on the
// device (the SM count bounds ctas and sets its default).
gmm_status host_fp8_config(int64_t N, int fuse, const gmm_fp8_tile_config* in, int sms, gmm_fp8_tile_config* out);
// Encodes the tensor maps and launches the FP8 forward with a resolved
// configuration, after the caller validated the arguments and, when needed,
// enqueued the group metadata into `workspace` (M > 0).  out: bf16 [M, N] or
// NULL (fused cast only); hq/hs: the fused FP8 cast of the output or NULL;
// w4: the weights are packed 4-bit E2M1 codes instead of e4m3.
gmm_status host_fp8_launch(const void* xq, const float* xs, const void* wq, const float* ws, int G, int64_t M,
                           int64_t K, int64_t N, int fuse, void* out, void* hq, float* hs, void* workspace,
                           const gmm_fp8_tile_config& cfg, cudaStream_t s, int w4);

}  // namespace gmm
