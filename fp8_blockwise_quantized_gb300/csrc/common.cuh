// Definitions shared by the kernels and the host launch layer.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
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
// Work counters of the CTA-pair tgmm kernel: units claimed, and CTAs that have
// finished (the last one resets both to zero for the next launch).
constexpr int kWsClaimed = 4;
constexpr int kWsFinished = 5;
// Number of 256-row tiles (the CTA-pair FP8 kernel's row tiles).
constexpr int kWsNumPairTiles = 6;
constexpr int kWsOffsets = 8;

// Row tile height of every grouped kernel (the tcgen05 MMA M).
constexpr int kBM = 128;
// Largest supported number of groups.
constexpr int kMaxGroups = 4096;

__host__ __device__ inline int64_t tiles_capacity(int G, int64_t M) { return (M + kBM - 1) / kBM + G; }
__host__ __device__ inline int64_t tiles_offset_bytes(int G) {
  return ((static_cast<int64_t>(kWsOffsets + G + 1) * 4 + 15) / 16) * 16;
}
// the groups ordered by size (descending, ties by index) follow the tiles
__host__ __device__ inline int64_t order_offset_bytes(int G, int64_t M) {
  return tiles_offset_bytes(G) + 16 * tiles_capacity(G, M);
}
// then the 256-row tiles of every group (the CTA-pair FP8 kernel's tiles)
__host__ __device__ inline int64_t pair_tiles_capacity(int G, int64_t M) { return (M + 2 * kBM - 1) / (2 * kBM) + G; }
__host__ __device__ inline int64_t pair_tiles_offset_bytes(int G, int64_t M) {
  return order_offset_bytes(G, M) + ((4 * static_cast<int64_t>(G) + 15) / 16) * 16;
}
__host__ __device__ inline int64_t workspace_bytes(int G, int64_t M) {
  return pair_tiles_offset_bytes(G, M) + 16 * pair_tiles_capacity(G, M);
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

// Per-block quantization arithmetic ("实现差距：GMM Kernel（V1 vs V2）", §3.3):
// scale = absmax / 448 and inv = (scale == 0 ? 0 : 1 / scale), both IEEE fp32
// round-to-nearest divisions; codes = e4m3(x * inv), nearest-even, saturating.
// Shared by the quantize kernels and the fused epilogue so that both produce
// the same bits.
__device__ __forceinline__ void e4m3_block_scale(float absmax, float& s, float& inv) {
  s = __fdiv_rn(absmax, 448.0f);
  inv = (s == 0.0f) ? 0.0f : __fdiv_rn(1.0f, s);
}
// The same block rule for 4-bit E2M1 weight codes, whose largest value is 6
// ("实现差距：GMM Kernel（V1 vs V2）", §3.4: 4-bit weight types with the
// blockwise fp32 scales kept): scale = absmax / 6, inv = (scale == 0 ? 0 :
// 1 / scale).
__device__ __forceinline__ void e2m1_block_scale(float absmax, float& s, float& inv) {
  s = __fdiv_rn(absmax, 6.0f);
  inv = (s == 0.0f) ? 0.0f : __fdiv_rn(1.0f, s);
}
// 2 x fp32 -> 2 x e4m3; `lo` is the lower byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// max |v| over the 8 bf16 values of a 16-byte chunk
__device__ __forceinline__ float bf16x8_absmax(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xffff0000u))));
  return m;
}
// 8 bf16 values (a 16-byte chunk) -> 8 e4m3 codes: e4m3(fp32(v) * inv)
__device__ __forceinline__ uint2 bf16x8_to_e4m3(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t q[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t p0 = w[2 * i], p1 = w[2 * i + 1];
    q[i] = e4m3x2(__fmul_rn(__uint_as_float(p0 << 16), inv), __fmul_rn(__uint_as_float(p0 & 0xffff0000u), inv)) |
           (e4m3x2(__fmul_rn(__uint_as_float(p1 << 16), inv), __fmul_rn(__uint_as_float(p1 & 0xffff0000u), inv))
            << 16);
  }
  return make_uint2(q[0], q[1]);
}

// silu(v) = v / (1 + exp(-v)), with the fast hardware exponential and divide
// (relative error a few ulp of fp32, far below the bf16 rounding that
// follows).  Saturates correctly: exp(-v) = inf gives 0.
__device__ __forceinline__ float silu_f32(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// Warp-cooperative store of up to 32 staged rows: row i of the warp lives at
// stage + i * STRIDE (ROW_BYTES bytes, a multiple of 16) and goes to
// gdst + i * ld_bytes; rows i >= nvalid are skipped.  Every store
// instruction writes 512 contiguous bytes per 256-byte pair of rows (or four
// 128-byte rows), so the output is written in whole cache lines.
template <int ROW_BYTES, int STRIDE>
__device__ __forceinline__ void warp_store_rows(const uint8_t* stage, uint8_t* gdst, long long ld_bytes,
                                                int nvalid, int lane) {
  constexpr int CPR = ROW_BYTES / 16;  // 16-byte chunks per row
  static_assert(CPR >= 1 && CPR <= 32 && (32 % CPR) == 0, "row size");
  constexpr int RPI = 32 / CPR;        // rows per instruction
  const int c = lane % CPR;
#pragma unroll
  for (int it = 0; it < 32 / RPI; ++it) {
    const int r = it * RPI + lane / CPR;
    if (r < nvalid)
      *reinterpret_cast<uint4*>(gdst + r * ld_bytes + c * 16) =
          *reinterpret_cast<const uint4*>(stage + r * STRIDE + c * 16);
  }
}

}  // namespace gmm
