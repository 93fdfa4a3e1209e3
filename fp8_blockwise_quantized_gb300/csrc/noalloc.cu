// gmm_fp8_fwd_noalloc: the FP8 grouped forward for callers that cannot hand
// the library a workspace.
//
// Some callers cannot call cudaMalloc at the point where they run the layer:
// code inside a framework whose allocator owns all device memory, a runtime
// that must not allocate after start-up (fixed memory budgets, real-time
// loops), or a plug-in that only receives its input and output pointers.
// This entry point needs nothing but those: the group metadata that the
// grouped kernels read lives in a fixed-size array in the library's own
// device memory (a file-scope __device__ variable), which the CUDA module
// loader reserves on every GPU that loads the library and keeps until the
// process exits.  Nothing is allocated per call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gmm.h"
#include "common.cuh"
#include "host.cuh"
#include "kernels.cuh"

using namespace gmm;

namespace {

// Static scratch: status word, group offsets and the row-tile lists of one
// call.  64 KiB covers, for example, G <= 1024 groups with M <= 65536 rows or
// G <= 256 with M <= 262144; the exact rule is gmm_workspace_bytes(G, M) <=
// kNoAllocScratchBytes.
constexpr size_t kNoAllocScratchBytes = 64 * 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Per-device set-up, done by the first call on each device with that device
// current: the device address of the static scratch (in host code the
// variable's name is only a host-side stand-in, never a device address) and
// the SM count.
struct NoAllocDevice {
  void* scratch = nullptr;
  int sms = 0;
  bool ready = false;
};

gmm_status noalloc_setup(NoAllocDevice* out) {
  static NoAllocDevice cache[64];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return host_cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return host_fail(GMM_ERR_UNSUPPORTED, "device ordinal beyond 63");
  std::lock_guard<std::mutex> lk(mu);
  NoAllocDevice& d = cache[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return host_cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) return host_fail(GMM_ERR_UNSUPPORTED, "the current device is not sm_103");
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return host_cuda_fail(e, "cudaGetSymbolAddress of the static scratch");
    if (ptr == nullptr) return host_fail(GMM_ERR_CUDA, "cudaGetSymbolAddress returned NULL");
    d.scratch = ptr;
    d.sms = sms;
    d.ready = true;
  }
  *out = d;
  return GMM_OK;
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" gmm_status gmm_fp8_fwd_noalloc(const void* xq, const float* xs, const void* wq, const float* ws,
                                          const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N,
                                          int fuse_silu_mul, void* out, void* stream) {
  const int fuse = fuse_silu_mul ? 1 : 0;
  const int64_t Nw = fuse ? 2 * N : N;
  if (G < 1 || G > kMaxGroups || M < 0 || M > INT32_MAX || K < 128 || K % 128 != 0 || N < 128 || N % 128 != 0 ||
      K > (1 << 24) || N > (1 << 24) || static_cast<int64_t>(G) * Nw > INT32_MAX)
    return GMM_ERR_SHAPE;
  // sizes whose metadata does not fit the static scratch are refused
  if (static_cast<size_t>(workspace_bytes(G, M)) > kNoAllocScratchBytes) return GMM_ERR_WORKSPACE;
  if (!wq || !ws || !group_sizes) return GMM_ERR_NULL;
  if (M > 0 && (!xq || !xs || !out)) return GMM_ERR_NULL;
  if (!a16(xq) || !a16(xs) || !a16(wq) || !a16(ws) || !a16(out) || !a16(group_sizes)) return GMM_ERR_ALIGN;

  NoAllocDevice d;
  gmm_status st = noalloc_setup(&d);
  if (st != GMM_OK) return st;
  // the tile configuration gmm_fp8_fwd uses (the defaults), so that both
  // entry points run the same kernel and give the same bits
  gmm_fp8_tile_config cfg;
  if ((st = host_fp8_config(N, fuse, nullptr, d.sms, &cfg)) != GMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The scratch keeps whatever the previous call left; only the sticky error
  // word must start at zero (every other field is rewritten below).
  int32_t* meta = static_cast<int32_t*>(d.scratch);
  cudaError_t e = cudaMemsetAsync(meta + kWsStatus, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return host_cuda_fail(e, "clearing the static scratch's error word");
  e = launch_group_metadata(group_sizes, G, static_cast<int>(M), d.scratch, s);
  if (e != cudaSuccess) return host_cuda_fail(e, "group_metadata_kernel launch");
  if (M == 0) return GMM_OK;
  return host_fp8_launch(xq, xs, wq, ws, G, M, K, N, fuse, out, nullptr, nullptr, d.scratch, cfg, s, 0);
}
