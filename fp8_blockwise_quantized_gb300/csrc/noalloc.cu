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

// Static scratch: status word, group offsets and the row-tile list of one
// call.  64 KiB covers, for example, G <= 1024 groups with M <= 262144 rows;
// the exact rule is gmm_workspace_bytes(G, M) <= kNoAllocScratchBytes.
constexpr size_t kNoAllocScratchBytes = 64 * 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Per-device set-up, done by the first call on each device with that device
// current: the device address of the static scratch (in host code the
// variable's name is only a host-side stand-in, never a device address), the
// SM count, and the tensor-map encoder.
struct NoAllocDevice {
  void* scratch = nullptr;
  int sms = 0;
  bool ready = false;
};

gmm_status noalloc_setup(NoAllocDevice* out, EncodeTiledFn* encode) {
  static NoAllocDevice cache[64];
  static EncodeTiledFn fn = nullptr;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return host_cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return host_fail(GMM_ERR_UNSUPPORTED, "device ordinal beyond 63");
  std::lock_guard<std::mutex> lk(mu);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return host_cuda_fail(e, "looking up cuTensorMapEncodeTiled");
    if (q != cudaDriverEntryPointSuccess) return host_fail(GMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
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
  *encode = fn;
  return GMM_OK;
}

gmm_status encode(EncodeTiledFn fn, CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                  uint32_t box_inner, uint32_t box_outer, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8,
                  uint64_t elem_bytes = 1) {
  cuuint64_t dims[2] = {inner, outer < 1 ? 1 : outer};
  cuuint64_t strides[1] = {inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GMM_OK : host_fail(GMM_ERR_CUDA, "cuTensorMapEncodeTiled failed");
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
  EncodeTiledFn fn = nullptr;
  gmm_status st = noalloc_setup(&d, &fn);
  if (st != GMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The scratch keeps whatever the previous call left; only the sticky error
  // word must start at zero (every other field is rewritten below).
  int32_t* meta = static_cast<int32_t*>(d.scratch);
  cudaError_t e = cudaMemsetAsync(meta + kWsStatus, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return host_cuda_fail(e, "clearing the static scratch's error word");
  Tile* tiles = reinterpret_cast<Tile*>(static_cast<char*>(d.scratch) + tiles_offset_bytes(G));
  int32_t* order = reinterpret_cast<int32_t*>(static_cast<char*>(d.scratch) + order_offset_bytes(G, M));
  e = launch_pdl(group_metadata_kernel, dim3(1), dim3(1024), 0, s, group_sizes, G, static_cast<int>(M), meta, tiles,
                 order);
  if (e != cudaSuccess) return host_cuda_fail(e, "group_metadata_kernel launch");
  if (M == 0) return GMM_OK;

  const Fp8Geometry geo = fp8_geometry(static_cast<int>(N), fuse);
  CUtensorMap map_a, map_b, map_out;
  if ((st = encode(fn, &map_a, xq, K, M, 128, 128)) != GMM_OK) return st;
  if ((st = encode(fn, &map_b, wq, K, G * Nw, 128, geo.b_box_rows)) != GMM_OK) return st;
  if ((st = encode(fn, &map_out, out, N, M, 64, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2)) != GMM_OK) return st;
  FwdArgs a{};
  a.xs = xs;
  a.ws = ws;
  a.meta = meta;
  a.tiles = tiles;
  a.out = static_cast<uint16_t*>(out);
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.fuse = fuse;
  a.wait_limit_ns = host_wait_limit_ns();
  const long long max_units = tiles_capacity(G, M) * (N / geo.out_cols);
  if (max_units >= (1LL << 31)) return GMM_ERR_SHAPE;  // the kernel's unit indices are 32-bit
  const int grid = static_cast<int>(max_units < d.sms ? max_units : d.sms);
  e = launch_gmm_fp8(map_a, map_b, map_out, a, grid, s);
  return e == cudaSuccess ? GMM_OK : host_cuda_fail(e, "gmm_fp8 kernel launch");
}
