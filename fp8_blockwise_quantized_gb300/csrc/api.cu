// Host side of the C ABI declared in include/gmm.h: argument validation,
// TMA tensor-map encoding, grid sizing and kernel launches.  Nothing here
// allocates device memory or synchronizes, except gmm_get_device_status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gmm.h"
#include "common.cuh"
#include "host.cuh"
#include "kernels.cuh"

using namespace gmm;

namespace {
thread_local char g_last_error[256] = "no error";
}  // namespace

namespace gmm {

gmm_status host_cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", what, cudaGetErrorString(e));
  return GMM_ERR_CUDA;
}

gmm_status host_fail(gmm_status status, const char* what) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s", what);
  return status;
}

uint64_t host_wait_limit_ns() {
  static uint64_t v = []() -> uint64_t {
    const char* s = std::getenv("GMM_WAIT_LIMIT_MS");
    if (s && *s) {
      long long ms = std::atoll(s);
      if (ms > 0) return static_cast<uint64_t>(ms) * 1000000ull;
    }
    return static_cast<uint64_t>(kDefaultWaitLimitNs);
  }();
  return v;
}

}  // namespace gmm

namespace {

gmm_status cuda_fail(cudaError_t e, const char* what) { return host_cuda_fail(e, what); }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

gmm_status device_info(DeviceInfo* out) {
  static DeviceInfo cache[64];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return GMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev].ok) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      std::snprintf(g_last_error, sizeof g_last_error, "device %d is sm_%d%d, the library is built for sm_103a", dev,
                    major, minor);
      return GMM_ERR_UNSUPPORTED;
    }
    cache[dev].sms = sms;
    cache[dev].ok = true;
  }
  *out = cache[dev];
  return GMM_OK;
}

uint64_t wait_limit_ns() { return host_wait_limit_ns(); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gmm_status encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
                     uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled is not available");
    return GMM_ERR_CUDA;
  }
  cuuint64_t dims[2] = {inner, outer < 1 ? 1 : outer};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return GMM_ERR_CUDA;
  }
  return GMM_OK;
}

// Tensor map of packed 4-bit weight codes: `rows` rows of K codes (K/2 bytes),
// boxes of 128 codes x box_rows rows, each 16 codes landing in 16 bytes of
// shared memory (the 4-bit MMA operand layout), 128-byte swizzle.  The base
// must be 32-byte aligned and K a multiple of 128 (the rows' stride a
// multiple of 32 bytes).
gmm_status encode_2d_w4(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled is not available");
    return GMM_ERR_CUDA;
  }
  cuuint64_t dims[2] = {K, rows < 1 ? 1 : rows};
  cuuint64_t strides[1] = {K / 2};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled (4-bit weights) failed (%d)",
                  static_cast<int>(r));
    return GMM_ERR_CUDA;
  }
  return GMM_OK;
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Shape checks shared by the grouped calls.
gmm_status check_grouped(int G, int64_t M, int64_t K, int64_t N, int64_t Nw) {
  if (G < 1 || G > kMaxGroups) return GMM_ERR_SHAPE;
  if (M < 0 || M > INT32_MAX) return GMM_ERR_SHAPE;
  if (K < 128 || K % 128 != 0 || N < 128 || N % 128 != 0) return GMM_ERR_SHAPE;
  if (K > (1 << 24) || N > (1 << 24)) return GMM_ERR_SHAPE;
  if (static_cast<int64_t>(G) * Nw > INT32_MAX || static_cast<int64_t>(G) * K > INT32_MAX) return GMM_ERR_SHAPE;
  return GMM_OK;
}

gmm_status launch_metadata(const int32_t* sizes, int G, int64_t M, void* workspace, cudaStream_t st) {
  cudaError_t e = launch_group_metadata(sizes, G, static_cast<int>(M), workspace, st);
  return e == cudaSuccess ? GMM_OK : cuda_fail(e, "group_metadata_kernel launch");
}

gmm_status check_workspace(const void* workspace, size_t bytes, int G, int64_t M) {
  if (!workspace) return GMM_ERR_WORKSPACE;
  if (!aligned16(workspace)) return GMM_ERR_ALIGN;
  if (bytes < static_cast<size_t>(workspace_bytes(G, M))) return GMM_ERR_WORKSPACE;
  return GMM_OK;
}

}  // namespace

namespace {

// The FP8 forward entry points: argument checks (all before any launch),
// the group metadata unless group_sizes is NULL, then the launch.  quant: the
// fused gate/up forward that also writes its output's 1x128 FP8 cast (hq, hs;
// out = h may be NULL); w4: 4-bit E2M1 weight codes, packed.
gmm_status fp8_entry(const void* xq, const float* xs, const void* wq, const float* ws, const int32_t* group_sizes,
                     int G, int64_t M, int64_t K, int64_t N, int fuse, void* out, void* hq, float* hs, bool quant,
                     void* workspace, size_t workspace_bytes, void* stream, const gmm_fp8_tile_config* config,
                     int w4);

}  // namespace

namespace gmm {

int host_fp8_default_cta_group(int64_t, int, int, int) {
  // one CTA per tile: on the production shapes the CTA-pair kernel measured
  // 316 / 171 us against 191 / 124 us (wi / wo); its N = 128 pair MMAs issue
  // far below their math rate
  return 1;
}

gmm_status host_fp8_config(int64_t N, int fuse, const gmm_fp8_tile_config* in, int sms, gmm_fp8_tile_config* out) {
  gmm_fp8_tile_config c = in ? *in : gmm_fp8_tile_config{0, 0, 0, 0, 0, 0};
  if (c.cta_group == 0) c.cta_group = host_fp8_default_cta_group(N, fuse, c.bn, c.ctas);
  if (c.cta_group != 1 && c.cta_group != 2) return GMM_ERR_UNSUPPORTED;
  if (c.bn != 0 && c.bn != 128 && c.bn != 256) return GMM_ERR_UNSUPPORTED;
  if (c.ctas < 0 || (sms > 0 && c.ctas > sms) || c.unit_order < 0 || c.unit_order > 2) return GMM_ERR_UNSUPPORTED;
  if (c.cta_group == 2) {
    // units of 256 weight columns (two MMA halves of 128): 128 gate + 128 up
    // columns when fused, else 256 output columns
    if (c.bn == 128 || (!fuse && N % 256 != 0)) return GMM_ERR_UNSUPPORTED;
    if (c.ctas % 2 != 0) return GMM_ERR_UNSUPPORTED;
    c.bn = 256;
  } else {
    if (c.bn == 256 && N % 256 != 0) return GMM_ERR_UNSUPPORTED;
    if (c.bn == 128 && fuse) return GMM_ERR_UNSUPPORTED;
    if (c.bn == 0) c.bn = (fuse || N % 256 == 0) ? 256 : 128;
  }
  if (c.ctas == 0) c.ctas = c.cta_group == 2 ? sms - sms % 2 : sms;
  if (c.unit_order == 0) c.unit_order = 1;
  // compiled instances: ring slots and TMEM partial buffers
  int smin, smax, sdef, bdef;
  bool bufs_ok;
  if (c.cta_group == 2) {
    smin = 3, smax = fuse ? 5 : 4, sdef = smax, bdef = 4;
    bufs_ok = c.tmem_bufs == 0 || c.tmem_bufs == 4;
  } else if (c.bn == 256) {
    smin = 2, smax = 3, sdef = 3, bdef = 2;
    bufs_ok = c.tmem_bufs == 0 || c.tmem_bufs == 2;
  } else {
    smin = 3, smax = 5, sdef = 4, bdef = 2;
    bufs_ok = c.tmem_bufs == 0 || c.tmem_bufs == 2 || c.tmem_bufs == 4;
  }
  if (c.stages != 0 && (c.stages < smin || c.stages > smax)) return GMM_ERR_UNSUPPORTED;
  if (!bufs_ok) return GMM_ERR_UNSUPPORTED;
  if (c.stages == 0) c.stages = sdef;
  if (c.tmem_bufs == 0) c.tmem_bufs = bdef;
  *out = c;
  return GMM_OK;
}

gmm_status host_fp8_launch(const void* xq, const float* xs, const void* wq, const float* ws, int G, int64_t M,
                           int64_t K, int64_t N, int fuse, void* out, void* hq, float* hs, void* workspace,
                           const gmm_fp8_tile_config& cfg, cudaStream_t s, int w4) {
  const bool pair = cfg.cta_group == 2;
  const int64_t Nw = fuse ? 2 * N : N;
  // MMA N per unit, output columns per unit, rows of the weight tensor-map box
  const Fp8Geometry geo = pair ? Fp8Geometry{128, fuse ? 128 : 256, 64} : fp8_geometry(static_cast<int>(N), fuse, cfg.bn);
  CUtensorMap map_a, map_b, map_out;
  gmm_status st;
  if ((st = encode_2d(&map_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xq, K, M, 128, 128)) != GMM_OK) return st;
  if (w4) {
    // packed 4-bit codes [G*Nw][K/2] bytes, expanded by the copy into the
    // shared-memory layout of 4-bit MMA operands (16 codes in each 16 bytes)
    if ((st = encode_2d_w4(&map_b, wq, K, G * Nw, geo.b_box_rows)) != GMM_OK) return st;
  } else if ((st = encode_2d(&map_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wq, K, G * Nw, 128, geo.b_box_rows)) !=
             GMM_OK) {
    return st;
  }
  // the bf16 output is written through its own tensor map; the fused cast
  // without h stores only hq and hs and never reads map_out
  if (out) {
    if ((st = encode_2d(&map_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, N, M, 64, 32)) != GMM_OK) return st;
  } else {
    map_out = map_a;
  }
  FwdArgs a{};
  a.xs = xs;
  a.ws = ws;
  a.meta = static_cast<const int32_t*>(workspace);
  a.tiles = reinterpret_cast<const Tile*>(static_cast<const char*>(workspace) + tiles_offset_bytes(G));
  a.pair_tiles = reinterpret_cast<const Tile*>(static_cast<const char*>(workspace) + pair_tiles_offset_bytes(G, M));
  a.out = static_cast<uint16_t*>(out);
  a.hq = static_cast<uint8_t*>(hq);
  a.hs = hs;
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.fuse = fuse;
  a.bn = geo.bn_mma;
  a.col_major = cfg.unit_order == 2 ? 1 : 0;
  a.b_fmt = w4 ? 5 : 0;  // kind::f8f6f4 operand types: e2m1 or e4m3
  a.stages = cfg.stages;
  a.tmem_bufs = cfg.tmem_bufs;
  a.wait_limit_ns = host_wait_limit_ns();
  const long long tiles = pair ? pair_tiles_capacity(G, M) : tiles_capacity(G, M);
  const long long max_units = tiles * (N / geo.out_cols);
  if (max_units >= (1LL << 31)) return GMM_ERR_SHAPE;  // the kernels' unit indices are 32-bit
  cudaError_t e;
  if (pair) {
    const long long pairs = cfg.ctas / 2;
    e = launch_gmm_fp8_pair(map_a, map_b, map_out, a, static_cast<int>(max_units < pairs ? max_units : pairs), s);
  } else {
    e = launch_gmm_fp8(map_a, map_b, map_out, a, static_cast<int>(max_units < cfg.ctas ? max_units : cfg.ctas), s);
  }
  return e == cudaSuccess ? GMM_OK : host_cuda_fail(e, "gmm_fp8 kernel launch");
}

}  // namespace gmm

namespace {

gmm_status fp8_entry(const void* xq, const float* xs, const void* wq, const float* ws, const int32_t* group_sizes,
                     int G, int64_t M, int64_t K, int64_t N, int fuse, void* out, void* hq, float* hs, bool quant,
                     void* workspace, size_t workspace_bytes, void* stream, const gmm_fp8_tile_config* config,
                     int w4) {
  const int64_t Nw = fuse ? 2 * N : N;
  gmm_status st = check_grouped(G, M, K, N, Nw);
  if (st != GMM_OK) return st;
  if (!wq || !ws) return GMM_ERR_NULL;
  if (M > 0 && (!xq || !xs)) return GMM_ERR_NULL;
  if (M > 0 && (quant ? (!hq || !hs) : !out)) return GMM_ERR_NULL;
  if (!aligned16(wq) || !aligned16(ws) || !aligned16(xq) || !aligned16(xs) || !aligned16(out) ||
      !aligned16(hq) || !aligned16(hs) || !aligned16(group_sizes))
    return GMM_ERR_ALIGN;
  if (w4 && !aligned32(wq)) return GMM_ERR_ALIGN;  // the 4-bit tensor map's base
  gmm_fp8_tile_config cfg;
  if ((st = host_fp8_config(N, fuse, config, 0, &cfg)) != GMM_OK) return st;  // the device-independent rules
  if (quant && cfg.bn != 256) return GMM_ERR_UNSUPPORTED;
  if ((st = check_workspace(workspace, workspace_bytes, G, M)) != GMM_OK) return st;
  DeviceInfo di;
  if ((st = device_info(&di)) != GMM_OK) return st;
  if ((st = host_fp8_config(N, fuse, config, di.sms, &cfg)) != GMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (group_sizes && (st = launch_metadata(group_sizes, G, M, workspace, s)) != GMM_OK) return st;
  if (M == 0) return GMM_OK;
  return host_fp8_launch(xq, xs, wq, ws, G, M, K, N, fuse, out, quant ? hq : nullptr, quant ? hs : nullptr,
                         workspace, cfg, s, w4);
}

}  // namespace

extern "C" {

const char* gmm_status_string(gmm_status s) {
  switch (s) {
    case GMM_OK: return "GMM_OK";
    case GMM_ERR_NULL: return "GMM_ERR_NULL: a required pointer is NULL";
    case GMM_ERR_SHAPE: return "GMM_ERR_SHAPE: a size is out of range or not a multiple of 128";
    case GMM_ERR_ALIGN: return "GMM_ERR_ALIGN: a pointer is not 16-byte aligned";
    case GMM_ERR_UNSUPPORTED: return "GMM_ERR_UNSUPPORTED: no sm_103 device is current";
    case GMM_ERR_CUDA: return "GMM_ERR_CUDA: a CUDA call failed";
    case GMM_ERR_GROUP_SIZES: return "GMM_ERR_GROUP_SIZES: a negative group size or sum(group_sizes) > M";
    case GMM_ERR_TIMEOUT: return "GMM_ERR_TIMEOUT: a kernel's bounded wait ran out";
    case GMM_ERR_WORKSPACE: return "GMM_ERR_WORKSPACE: workspace missing or too small";
  }
  return "unknown gmm_status";
}

const char* gmm_last_cuda_error(void) { return g_last_error; }

size_t gmm_workspace_bytes(int G, int64_t M) {
  if (G < 1 || M < 0) return 0;
  return static_cast<size_t>(workspace_bytes(G, M));
}

size_t gmm_tiles_offset(int G) { return G < 1 ? 0 : static_cast<size_t>(tiles_offset_bytes(G)); }

gmm_status gmm_group_metadata(const int32_t* group_sizes, int G, int64_t M, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!group_sizes) return GMM_ERR_NULL;
  if (G < 1 || G > kMaxGroups || M < 0 || M > INT32_MAX) return GMM_ERR_SHAPE;
  gmm_status st = check_workspace(workspace, workspace_bytes, G, M);
  if (st != GMM_OK) return st;
  DeviceInfo di;
  if ((st = device_info(&di)) != GMM_OK) return st;
  return launch_metadata(group_sizes, G, M, workspace, static_cast<cudaStream_t>(stream));
}

gmm_status gmm_quantize_lhs(const void* x, int64_t M, int64_t K, void* xq, float* xs, void* stream) {
  if (M < 0 || M > INT32_MAX || K < 128 || K % 128 != 0 || K > (1 << 24)) return GMM_ERR_SHAPE;
  if (M == 0) return GMM_OK;
  if (!x || !xq || !xs) return GMM_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(xs)) return GMM_ERR_ALIGN;
  DeviceInfo di;
  gmm_status st = device_info(&di);
  if (st != GMM_OK) return st;
  const long long nblocks = M * (K / 128);
  const long long per_cta = 8LL * kLhsBlocksPerWarp;  // 8 warps per CTA
  long long grid = (nblocks + per_cta - 1) / per_cta;
  if (grid > static_cast<long long>(di.sms) * 8) grid = static_cast<long long>(di.sms) * 8;
  cudaError_t e = launch_pdl(quantize_lhs_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                             static_cast<cudaStream_t>(stream), static_cast<const uint4*>(x), static_cast<int>(M),
                             static_cast<int>(K / 128), nblocks, static_cast<uint2*>(xq), xs);
  return e == cudaSuccess ? GMM_OK : cuda_fail(e, "quantize_lhs_kernel launch");
}

gmm_status gmm_quantize_rhs(const void* w, int G, int64_t K, int64_t N, void* wq, float* ws, void* stream) {
  if (G < 1 || K < 128 || K % 128 != 0 || N < 128 || N % 128 != 0 || K > (1 << 24) || N > (1 << 24))
    return GMM_ERR_SHAPE;
  if (static_cast<int64_t>(G) * (K / 128) * (N / 128) > INT32_MAX) return GMM_ERR_SHAPE;
  if (!w || !wq || !ws) return GMM_ERR_NULL;
  if (!aligned16(w) || !aligned16(wq) || !aligned16(ws)) return GMM_ERR_ALIGN;
  DeviceInfo di;
  gmm_status st = device_info(&di);
  if (st != GMM_OK) return st;
  const int grid = static_cast<int>(static_cast<int64_t>(G) * (K / 128) * (N / 128));
  quantize_rhs_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(w), static_cast<int>(K), static_cast<int>(N), static_cast<uint8_t*>(wq), ws);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GMM_OK : cuda_fail(e, "quantize_rhs_kernel launch");
}

gmm_status gmm_fp8_fwd(const void* xq, const float* xs, const void* wq, const float* ws, const int32_t* group_sizes,
                       int G, int64_t M, int64_t K, int64_t N, int fuse_silu_mul, void* out, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return fp8_entry(xq, xs, wq, ws, group_sizes, G, M, K, N, fuse_silu_mul ? 1 : 0, out, nullptr, nullptr, false,
                   workspace, workspace_bytes, stream, nullptr, 0);
}

gmm_status gmm_fp8_fwd_tiled(const void* xq, const float* xs, const void* wq, const float* ws,
                             const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N, int fuse_silu_mul,
                             void* out, void* workspace, size_t workspace_bytes, void* stream,
                             const gmm_fp8_tile_config* config) {
  return fp8_entry(xq, xs, wq, ws, group_sizes, G, M, K, N, fuse_silu_mul ? 1 : 0, out, nullptr, nullptr, false,
                   workspace, workspace_bytes, stream, config, 0);
}

gmm_status gmm_fp8_fwd_swiglu_quant(const void* xq, const float* xs, const void* wq, const float* ws,
                                    const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N, void* h,
                                    void* hq, float* hs, void* workspace, size_t workspace_bytes, void* stream) {
  return fp8_entry(xq, xs, wq, ws, group_sizes, G, M, K, N, 1, h, hq, hs, true, workspace, workspace_bytes, stream,
                   nullptr, 0);
}

gmm_status gmm_fp8_fwd_swiglu_quant_tiled(const void* xq, const float* xs, const void* wq, const float* ws,
                                          const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N,
                                          void* h, void* hq, float* hs, void* workspace, size_t workspace_bytes,
                                          void* stream, const gmm_fp8_tile_config* config) {
  return fp8_entry(xq, xs, wq, ws, group_sizes, G, M, K, N, 1, h, hq, hs, true, workspace, workspace_bytes, stream,
                   config, 0);
}

gmm_status gmm_quantize_rhs_w4(const void* w, int G, int64_t K, int64_t N, void* wq4, float* ws, void* stream) {
  if (G < 1 || K < 128 || K % 128 != 0 || N < 128 || N % 128 != 0 || K > (1 << 24) || N > (1 << 24))
    return GMM_ERR_SHAPE;
  if (static_cast<int64_t>(G) * (K / 128) * (N / 128) > INT32_MAX) return GMM_ERR_SHAPE;
  if (!w || !wq4 || !ws) return GMM_ERR_NULL;
  if (!aligned16(w) || !aligned32(wq4) || !aligned16(ws)) return GMM_ERR_ALIGN;
  DeviceInfo di;
  gmm_status st = device_info(&di);
  if (st != GMM_OK) return st;
  const int grid = static_cast<int>(static_cast<int64_t>(G) * (K / 128) * (N / 128));
  quantize_rhs_w4_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(w), static_cast<int>(K), static_cast<int>(N), static_cast<uint8_t*>(wq4), ws);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GMM_OK : cuda_fail(e, "quantize_rhs_w4_kernel launch");
}

gmm_status gmm_fp8_w4_fwd(const void* xq, const float* xs, const void* wq4, const float* ws,
                          const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N, int fuse_silu_mul,
                          void* out, void* workspace, size_t workspace_bytes, void* stream,
                          const gmm_fp8_tile_config* config) {
  return fp8_entry(xq, xs, wq4, ws, group_sizes, G, M, K, N, fuse_silu_mul ? 1 : 0, out, nullptr, nullptr, false,
                   workspace, workspace_bytes, stream, config, 1);
}

gmm_status gmm_fp8_w4_fwd_swiglu_quant(const void* xq, const float* xs, const void* wq4, const float* ws,
                                       const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N, void* h,
                                       void* hq, float* hs, void* workspace, size_t workspace_bytes, void* stream,
                                       const gmm_fp8_tile_config* config) {
  return fp8_entry(xq, xs, wq4, ws, group_sizes, G, M, K, N, 1, h, hq, hs, true, workspace, workspace_bytes, stream,
                   config, 1);
}

gmm_status gmm_bf16_fwd(const void* x, const void* w, const int32_t* group_sizes, int G, int64_t M, int64_t K,
                        int64_t N, int fuse_silu_mul, void* out, void* workspace, size_t workspace_bytes,
                        void* stream) {
  const int fuse = fuse_silu_mul ? 1 : 0;
  const int64_t Nw = fuse ? 2 * N : N;
  gmm_status st = check_grouped(G, M, K, N, Nw);
  if (st != GMM_OK) return st;
  if (!w) return GMM_ERR_NULL;
  if (M > 0 && (!x || !out)) return GMM_ERR_NULL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(out) || !aligned16(group_sizes)) return GMM_ERR_ALIGN;
  if ((st = check_workspace(workspace, workspace_bytes, G, M)) != GMM_OK) return st;
  DeviceInfo di;
  if ((st = device_info(&di)) != GMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (group_sizes && (st = launch_metadata(group_sizes, G, M, workspace, s)) != GMM_OK) return st;
  if (M == 0) return GMM_OK;

  const Fp8Geometry geo = bf16_geometry(static_cast<int>(N), fuse);
  CUtensorMap map_a, map_b;
  if ((st = encode_2d(&map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, K, M, 64, 128)) != GMM_OK) return st;
  if ((st = encode_2d(&map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, Nw, G * K, 64, 64)) != GMM_OK) return st;
  FwdArgs a{};
  a.meta = static_cast<const int32_t*>(workspace);
  a.tiles = reinterpret_cast<const Tile*>(static_cast<const char*>(workspace) + tiles_offset_bytes(G));
  a.out = static_cast<uint16_t*>(out);
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.fuse = fuse;
  a.wait_limit_ns = wait_limit_ns();
  const long long max_units = tiles_capacity(G, M) * (N / geo.out_cols);
  const int grid = static_cast<int>(max_units < di.sms ? max_units : di.sms);
  cudaError_t e = launch_gmm_bf16(map_a, map_b, a, grid, s);
  return e == cudaSuccess ? GMM_OK : cuda_fail(e, "gmm_bf16 kernel launch");
}

gmm_status gmm_bf16_dgrad(const void* dy, const void* w, const int32_t* group_sizes, int G, int64_t M, int64_t K,
                          int64_t N, void* dx, void* workspace, size_t workspace_bytes, void* stream) {
  // dX [M, K] = dY [M, N] . W[g]^T, W [G, K, N]: a grouped GEMM whose
  // reduction is N and whose output columns are K
  gmm_status st = check_grouped(G, M, N, K, K);
  if (st != GMM_OK) return st;
  if (!w) return GMM_ERR_NULL;
  if (M > 0 && (!dy || !dx)) return GMM_ERR_NULL;
  if (!aligned16(dy) || !aligned16(w) || !aligned16(dx) || !aligned16(group_sizes)) return GMM_ERR_ALIGN;
  if ((st = check_workspace(workspace, workspace_bytes, G, M)) != GMM_OK) return st;
  DeviceInfo di;
  if ((st = device_info(&di)) != GMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (group_sizes && (st = launch_metadata(group_sizes, G, M, workspace, s)) != GMM_OK) return st;
  if (M == 0) return GMM_OK;

  const int bn = (K % 256 == 0) ? 256 : 128;
  CUtensorMap map_a, map_b;
  if ((st = encode_2d(&map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dy, N, M, 64, 128)) != GMM_OK) return st;
  if ((st = encode_2d(&map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, N, static_cast<int64_t>(G) * K, 64, bn)) !=
      GMM_OK)
    return st;
  FwdArgs a{};
  a.meta = static_cast<const int32_t*>(workspace);
  a.tiles = reinterpret_cast<const Tile*>(static_cast<const char*>(workspace) + tiles_offset_bytes(G));
  a.out = static_cast<uint16_t*>(dx);
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(N);
  a.N = static_cast<int>(K);
  a.fuse = 0;
  a.wait_limit_ns = wait_limit_ns();
  const long long max_units = tiles_capacity(G, M) * (K / bn);
  const int grid = static_cast<int>(max_units < di.sms ? max_units : di.sms);
  cudaError_t e = launch_gmm_bf16_dgrad(map_a, map_b, a, grid, s);
  return e == cudaSuccess ? GMM_OK : cuda_fail(e, "gmm_bf16 dgrad kernel launch");
}

gmm_status tgmm_bf16(const void* x, const void* dy, const int32_t* group_sizes, int G, int64_t M, int64_t K,
                     int64_t N, void* dw, void* workspace, size_t workspace_bytes, void* stream) {
  return tgmm_bf16_tiled(x, dy, group_sizes, G, M, K, N, dw, workspace, workspace_bytes, stream, nullptr);
}

gmm_status tgmm_bf16_tiled(const void* x, const void* dy, const int32_t* group_sizes, int G, int64_t M, int64_t K,
                           int64_t N, void* dw, void* workspace, size_t workspace_bytes, void* stream,
                           const gmm_tgmm_tile_config* config) {
  gmm_status st = check_grouped(G, M, K, N, N);
  if (st != GMM_OK) return st;
  gmm_tgmm_tile_config cfg = config ? *config : gmm_tgmm_tile_config{0, 0, 0};
  if (cfg.stages != 0 && (cfg.stages < 4 || cfg.stages > 6)) return GMM_ERR_UNSUPPORTED;
  if (cfg.claim_ahead < 0 || cfg.claim_ahead > 12 || cfg.max_batch < 0 || cfg.max_batch > 4)
    return GMM_ERR_UNSUPPORTED;
  if (cfg.stages == 0) cfg.stages = 6;
  if (cfg.claim_ahead == 0) cfg.claim_ahead = 3;
  if (cfg.max_batch == 0) cfg.max_batch = 4;
  // the kernel walks its output tiles with 32-bit indices
  if (static_cast<int64_t>(G) * (K / 128) * (N / tgmm_bn(static_cast<int>(N))) > INT32_MAX / 2) return GMM_ERR_SHAPE;
  if (!dw) return GMM_ERR_NULL;
  if (M > 0 && (!x || !dy)) return GMM_ERR_NULL;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dw) || !aligned16(group_sizes)) return GMM_ERR_ALIGN;
  if ((st = check_workspace(workspace, workspace_bytes, G, M)) != GMM_OK) return st;
  DeviceInfo di;
  if ((st = device_info(&di)) != GMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (group_sizes && (st = launch_metadata(group_sizes, G, M, workspace, s)) != GMM_OK) return st;

  // With M == 0 every group is empty: the kernel only writes zeros and never
  // reads x or dy, so the maps may describe a dummy one-row tensor.
  const void* xb = M > 0 ? x : dw;
  const void* db = M > 0 ? dy : dw;
  CUtensorMap map_x, map_dy, map_dw;
  if ((st = encode_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xb, K, M, 64, 64)) != GMM_OK) return st;
  if ((st = encode_2d(&map_dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, db, N, M, 64, 64)) != GMM_OK) return st;
  // dW viewed as [G*K, N], written in 32-row x 64-column boxes
  if ((st = encode_2d(&map_dw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dw, N, static_cast<int64_t>(G) * K, 64, 32)) !=
      GMM_OK)
    return st;
  TgmmArgs a{};
  a.meta = static_cast<const int32_t*>(workspace);
  a.order = reinterpret_cast<const int32_t*>(static_cast<const char*>(workspace) + order_offset_bytes(G, M));
  a.dw = static_cast<uint16_t*>(dw);
  a.G = G;
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.stages = cfg.stages;
  a.claim_ahead = cfg.claim_ahead;
  a.max_batch = cfg.max_batch;
  a.wait_limit_ns = wait_limit_ns();
  const long long units = static_cast<long long>(G) * (K / 128) * (N / tgmm_bn(static_cast<int>(N)));
  const int grid = static_cast<int>(units < di.sms ? units : di.sms);
  cudaError_t e = launch_tgmm_bf16(map_x, map_dy, map_dw, a, grid, s);
  return e == cudaSuccess ? GMM_OK : cuda_fail(e, "tgmm kernel launch");
}

gmm_status gmm_get_device_status(void* workspace, void* stream) {
  if (!workspace) return GMM_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace status word");
  if (word != 0) {
    e = cudaMemsetAsync(workspace, 0, sizeof word, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace status word");
  }
  if (word & kErrTimeout) return GMM_ERR_TIMEOUT;
  if (word & (kErrNegativeGroup | kErrGroupsExceedM)) return GMM_ERR_GROUP_SIZES;
  return GMM_OK;
}

}  // extern "C"
