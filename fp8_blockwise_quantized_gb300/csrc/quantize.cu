// a2 / a3: blockwise e4m3 quantization.
//
// Per block ("实现差距：GMM Kernel（V1 vs V2）", §3.3): absmax = max|x|,
// scale = absmax / 448, inv = (scale == 0 ? 0 : 1/scale), q = e4m3(x * inv).
// Block shapes ("GEMM Kernel 性能优化十问", Q2): 1x128 for the activations
// (one scale per row per 128 elements), 128x128 for the weights.
//
// The scale arithmetic is IEEE fp32 with round-to-nearest: __fdiv_rn and
// __fmul_rn keep the compiler from contracting or approximating it, so the
// codes and scales are bit-identical to any correct fp32 implementation.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace gmm {

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

}  // namespace

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// LHS, 1x128 blocks.  X is row-major [M, K] with K % 128 == 0; block (m, kb)
// occupies bytes [256 (m KB + kb), + 256) of X.  A half-warp (16 lanes x 16
// bytes) handles one block; a warp handles the blocks kb of eight consecutive
// rows per step (slots in groups of 8 rows), all loads issued before any
// reduction, for memory-level parallelism, so that its eight scales are one
// contiguous 32-byte run of xs[kb][m] instead of eight scattered words.
__global__ void __launch_bounds__(256) quantize_lhs_kernel(const uint4* __restrict__ x, int M, int KB,
                                                           long long nblocks, uint2* __restrict__ xq,
                                                           float* __restrict__ xs) {
  constexpr int kPerHalf = kLhsBlocksPerWarp / 2;
  static_assert(kLhsBlocksPerWarp == 8, "a warp step covers eight rows");
  (void)nblocks;
  griddep_launch_dependents();
  griddep_wait();  // x may come from the previous kernel
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;

  const long long nslots = ((M + 7) / 8) * 8LL * KB;
  for (long long base = warp_id * kLhsBlocksPerWarp; base < nslots; base += nwarps * kLhsBlocksPerWarp) {
    {
      // the warp's next step: its 16 lines (8 rows x 256 bytes) into L2 now,
      // so that the loads of that step find them there (one step ahead is
      // what helps; two steps ahead evicts lines before they are used)
      const long long nb = base + nwarps * kLhsBlocksPerWarp;
      if (lane < 16 && nb < nslots) {
        const long long g2 = nb >> 3;
        const long long m2 = (g2 / KB) * 8 + (lane >> 1), k2 = g2 - (g2 / KB) * KB;
        if (m2 < M) prefetch_l2(x + (m2 * KB + k2) * 16 + (lane & 1) * 8);
      }
    }
    uint4 v[kPerHalf];
    const long long grp = base >> 3;
    const long long mg = grp / KB, kbg = grp - mg * KB;
#pragma unroll
    for (int i = 0; i < kPerHalf; ++i) {
      const long long m = mg * 8 + half * kPerHalf + i;
      const long long b = m * KB + kbg;
      v[i] = (m < M) ? __ldcs(x + b * 16 + l16) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kPerHalf; ++i) {
      const long long m = mg * 8 + half * kPerHalf + i;
      const long long b = m * KB + kbg;
      float f[8];
      bf16x8_to_f32(v[i], f);
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
      for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
      float s, inv;
      e4m3_block_scale(amax, s, inv);
      uint2 q;
      q.x = e4m3x2(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv)) |
            (e4m3x2(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv)) << 16);
      q.y = e4m3x2(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv)) |
            (e4m3x2(__fmul_rn(f[6], inv), __fmul_rn(f[7], inv)) << 16);
      if (m < M) {
        xq[b * 16 + l16] = q;
        if (l16 == 0) xs[kbg * M + m] = s;
      }
    }
  }
}

// RHS, 128x128 blocks, offline.  One CTA of 256 threads per block (g, kb,
// nb): load the bf16 block, reduce its absmax, quantize, transpose through
// shared memory and write wq in the K-major layout [G][N][K].
__global__ void __launch_bounds__(256) quantize_rhs_kernel(const uint16_t* __restrict__ w, int K, int N,
                                                           uint8_t* __restrict__ wq, float* __restrict__ ws) {
  __shared__ float red[8];
  __shared__ uint8_t tile[128][128 + 16];  // [n][k], padded
  const int KB = K / 128, NB = N / 128;
  const int nb = blockIdx.x % NB;
  const int kb = (blockIdx.x / NB) % KB;
  const long long g = blockIdx.x / (static_cast<long long>(NB) * KB);
  const int t = threadIdx.x;
  // thread t covers row k = t/2 of the block, columns 64*(t%2) .. +64
  const int kr = t >> 1, c0 = (t & 1) * 64;
  const uint4* src = reinterpret_cast<const uint4*>(
      w + (g * K + static_cast<long long>(kb) * 128 + kr) * N + static_cast<long long>(nb) * 128 + c0);
  float f[64];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float e[8];
    bf16x8_to_f32(src[i], e);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[8 * i + j] = e[j];
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 64; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  if ((t & 31) == 0) red[t >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  float s, inv;
  e4m3_block_scale(amax, s, inv);
#pragma unroll
  for (int j = 0; j < 64; j += 2) {
    const uint32_t q = e4m3x2(__fmul_rn(f[j], inv), __fmul_rn(f[j + 1], inv));
    tile[c0 + j][kr] = static_cast<uint8_t>(q & 0xff);
    tile[c0 + j + 1][kr] = static_cast<uint8_t>(q >> 8);
  }
  __syncthreads();
  // write out: thread t -> output row n = t/2 of the block, 64 k-bytes
  const int nr = t >> 1, k0 = (t & 1) * 64;
  uint8_t* dst = wq + (g * N + static_cast<long long>(nb) * 128 + nr) * K + static_cast<long long>(kb) * 128 + k0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v;
    const uint8_t* p = &tile[nr][k0 + 16 * i];
    v.x = p[0] | (p[1] << 8) | (p[2] << 16) | (static_cast<uint32_t>(p[3]) << 24);
    v.y = p[4] | (p[5] << 8) | (p[6] << 16) | (static_cast<uint32_t>(p[7]) << 24);
    v.z = p[8] | (p[9] << 8) | (p[10] << 16) | (static_cast<uint32_t>(p[11]) << 24);
    v.w = p[12] | (p[13] << 8) | (p[14] << 16) | (static_cast<uint32_t>(p[15]) << 24);
    reinterpret_cast<uint4*>(dst)[i] = v;
  }
  if (t == 0) ws[(g * KB + kb) * NB + nb] = s;
}

// RHS, 128x128 blocks, 4-bit E2M1 codes, offline ("实现差距：GMM Kernel（V1 vs
// V2）", §3.4).  As quantize_rhs_kernel with scale = absmax / 6; the codes go
// out packed two per byte in the K-major layout [G][N][K/2]: byte k/2 of row
// n holds the code of k (even) in its low nibble and that of k + 1 in its
// high nibble, the order in which the tensor core reads 4-bit operands.
__global__ void __launch_bounds__(256) quantize_rhs_w4_kernel(const uint16_t* __restrict__ w, int K, int N,
                                                              uint8_t* __restrict__ wq4, float* __restrict__ ws) {
  __shared__ float red[8];
  __shared__ uint8_t tile[128][128 + 16];  // [n][k] codes, one per byte, padded
  const int KB = K / 128, NB = N / 128;
  const int nb = blockIdx.x % NB;
  const int kb = (blockIdx.x / NB) % KB;
  const long long g = blockIdx.x / (static_cast<long long>(NB) * KB);
  const int t = threadIdx.x;
  const int kr = t >> 1, c0 = (t & 1) * 64;
  const uint4* src = reinterpret_cast<const uint4*>(
      w + (g * K + static_cast<long long>(kb) * 128 + kr) * N + static_cast<long long>(nb) * 128 + c0);
  float f[64];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float e[8];
    bf16x8_to_f32(src[i], e);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[8 * i + j] = e[j];
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 64; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  if ((t & 31) == 0) red[t >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  float s, inv;
  e2m1_block_scale(amax, s, inv);
#pragma unroll
  for (int j = 0; j < 64; ++j)
    tile[c0 + j][kr] =
        static_cast<uint8_t>(__nv_cvt_float_to_fp4(__fmul_rn(f[j], inv), __NV_E2M1, cudaRoundNearest) & 0xF);
  __syncthreads();
  // write out: thread t -> output row n = t/2 of the block, 64 codes = 32 bytes
  const int nr = t >> 1, k0 = (t & 1) * 64;
  uint8_t* dst = wq4 + (g * N + static_cast<long long>(nb) * 128 + nr) * (K / 2) + static_cast<long long>(kb) * 64 +
                 k0 / 2;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t word[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint8_t* p = &tile[nr][k0 + 32 * i + 8 * q];
      word[q] = static_cast<uint32_t>(p[0] | (p[1] << 4)) | (static_cast<uint32_t>(p[2] | (p[3] << 4)) << 8) |
                (static_cast<uint32_t>(p[4] | (p[5] << 4)) << 16) | (static_cast<uint32_t>(p[6] | (p[7] << 4)) << 24);
    }
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(word[0], word[1], word[2], word[3]);
  }
  if (t == 0) ws[(g * KB + kb) * NB + nb] = s;
}

}  // namespace gmm
