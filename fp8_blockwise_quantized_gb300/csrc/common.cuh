// Definitions shared by the kernels and the host launch layer.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gmm {

// Sticky device error bits (workspace word 0).
constexpr int kErrNegativeGroup = 1;
constexpr int kErrGroupsExceedM = 2;
constexpr int kErrTimeout = 4;

// Workspace layout (int32 words), see gmm_group_metadata in gmm.h.
constexpr int kWsStatus = 0;
constexpr int kWsValid = 1;
constexpr int kWsS = 2;
constexpr int kWsNumTiles = 3;
constexpr int kWsOffsets = 8;

// Row tile height of every grouped kernel (the tcgen05 MMA M).
constexpr int kBM = 128;
// Largest supported number of groups.
constexpr int kMaxGroups = 4096;

__host__ __device__ inline int64_t tiles_capacity(int G, int64_t M) { return (M + kBM - 1) / kBM + G; }
__host__ __device__ inline int64_t tiles_offset_bytes(int G) {
  return ((static_cast<int64_t>(kWsOffsets + G + 1) * 4 + 15) / 16) * 16;
}
__host__ __device__ inline int64_t workspace_bytes(int G, int64_t M) {
  return tiles_offset_bytes(G) + 16 * tiles_capacity(G, M);
}

// Bounded-wait limit handed to every kernel (nanoseconds of %globaltimer).
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;

struct Tile {
  int g, row0, row1, pad;
};

// Shared epilogue helpers ----------------------------------------------------
// Two fp32 -> bf16 (round to nearest even); `lo` lands at the lower address.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu_f32(float v) { return v / (1.0f + expf(-v)); }

}  // namespace gmm
