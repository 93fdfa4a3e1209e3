// Kernel entry points and their host-side launchers (internal to the library).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "common.cuh"

namespace gmm {

// Launch with programmatic stream serialization (see griddep_wait): the kernel
// may start while the previous kernel on the stream finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- a1 metadata ------------------------------------------------------------
__global__ void group_metadata_kernel(const int32_t* sizes, int G, int M, int32_t* ws, Tile* tiles,
                                      int32_t* order, Tile* pair_tiles);
// Launches the metadata kernel into a workspace laid out for (G, M).
cudaError_t launch_group_metadata(const int32_t* sizes, int G, int M, void* workspace, cudaStream_t stream);

// ---- a2 / a3 quantization -----------------------------------------------------
constexpr int kLhsBlocksPerWarp = 8;
__global__ void quantize_lhs_kernel(const uint4* x, int M, int KB, long long nblocks, uint2* xq, float* xs);
__global__ void quantize_rhs_kernel(const uint16_t* w, int K, int N, uint8_t* wq, float* ws);
__global__ void quantize_rhs_w4_kernel(const uint16_t* w, int K, int N, uint8_t* wq4, float* ws);

// ---- grouped GEMMs ------------------------------------------------------------
// Arguments shared by the grouped forward kernels.
struct FwdArgs {
  const float* xs;        // fp32 [K/128][M] (FP8 only)
  const float* ws;        // fp32 [G][K/128][Nw/128] (FP8 only)
  const int32_t* meta;    // workspace words
  const Tile* tiles;      // workspace tile list (128-row tiles)
  const Tile* pair_tiles; // workspace 256-row tiles (CTA-pair FP8 kernel)
  uint16_t* out;          // bf16 [M][N] (may be null with hq)
  uint8_t* hq;            // fused quantized output: e4m3 [M][N] (null: none)
  float* hs;              // fused quantized output scales: fp32 [N/128][M]
  int M, K, N;            // N = output columns
  int fuse;               // 1: silu(gate) * up, W has 2N columns
  int bn;                 // FP8: columns of W per unit (0: by N)
  int col_major;          // FP8: units ordered column block major
  int b_fmt;              // FP8: weight code type in the MMA instruction descriptor
                          // (kind::f8f6f4: 0 = e4m3, 5 = e2m1)
  int stages;             // FP8: ring slots of the launched instance
  int tmem_bufs;          // FP8: TMEM partial buffers of the launched instance
  uint64_t wait_limit_ns;
};

struct TgmmArgs {
  const int32_t* meta;    // workspace words (offsets)
  const int32_t* order;   // workspace: groups by size, descending
  uint16_t* dw;           // bf16 [G][K][N]
  int G, M, K, N;
  int stages;             // CTA-pair kernel with 256-column units: ring slots (4..6)
  int claim_ahead;        // CTA-pair kernel: units claimed beyond the producer (1..12)
  int max_batch;          // CTA-pair kernel: most small units per claim (1..4)
  uint64_t wait_limit_ns;
};

// Host launchers: `grid` CTAs (persistent), on `stream`.  Return the launch error.
// map_out: the bf16 output (out, or h when fused) [M, N], box 64 columns x
// 32 rows, 128-byte swizzle; read only when args.out is not null.
cudaError_t launch_gmm_fp8(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                           const FwdArgs& args, int grid, cudaStream_t stream);
// The single-CTA kernel's BN = 128 instances (gmm_fp8_n128.cu).
cudaError_t launch_gmm_fp8_n128(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                                const FwdArgs& args, int grid, cudaStream_t stream);
// The CTA-pair FP8 kernel: map_b's box is 64 rows (half of a 128-column MMA
// half); at most max_pairs clusters of two CTAs.
cudaError_t launch_gmm_fp8_pair(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                                const FwdArgs& args, int max_pairs, cudaStream_t stream);
cudaError_t launch_gmm_bf16(const CUtensorMap& map_a, const CUtensorMap& map_b, const FwdArgs& args, int grid,
                            cudaStream_t stream);
// bf16 dgrad: the forward kernel with a K-major weight ([G*N_out, K] view);
// args.K = reduction length, args.N = output columns.
cudaError_t launch_gmm_bf16_dgrad(const CUtensorMap& map_a, const CUtensorMap& map_b, const FwdArgs& args,
                                  int grid, cudaStream_t stream);
cudaError_t launch_tgmm_bf16(const CUtensorMap& map_x, const CUtensorMap& map_dy, const CUtensorMap& map_dw,
                             const TgmmArgs& args, int grid, cudaStream_t stream);

// Tile geometry the host needs to build tensor maps and size grids.
struct Fp8Geometry {
  int bn_mma;      // MMA N (columns of W per stage)
  int out_cols;    // output columns per work unit
  int b_box_rows;  // rows of the W tensor-map box
};
Fp8Geometry fp8_geometry(int N, int fuse, int bn = 0);
Fp8Geometry bf16_geometry(int N, int fuse);
int tgmm_bn(int N);

}  // namespace gmm
