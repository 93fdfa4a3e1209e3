// a7: bf16 grouped GEMM forward, unquantized (the BF16 baseline of "GEMM
// Kernel 性能优化十问", Q7 and Q10 step 4): out[m, n] = bf16(sum_k x[m,k] *
// w[g][k,n]) with fp32 accumulation, optionally bf16(silu(gate) * up) with the
// gate/up weight of "实现差距：GMM Kernel（V1 vs V2）", §3.5.
//
// With BK = true the weight operand is K-major instead: the same kernel then
// computes the bf16 dgrad dX_g = dY_g W[g]^T (the "bwd" phase of "GEMM Kernel
// 性能优化十问" Q4, bf16 per Q5), with W [G][K][N] read as rows of the output
// columns, N (its contiguous dimension) being the reduction.
//
// Same skeleton as the FP8 kernel without promotion: the accumulator stays in
// TMEM for the whole K loop (two TMEM buffers so the epilogue of one unit
// overlaps the MMAs of the next).
//   warp 0     TMA: X tile 128 rows x 64 k (K-major) and W[g] tile 64 k x BN
//              (N contiguous: MN-major, BN/64 boxes of 64 columns) per stage.
//   warp 1     TMEM allocation; tcgen05.mma kind::f16 (bf16), M=128, N=BN,
//              K=16, four per stage.
//   warps 2-9  epilogue: tcgen05.ld -> bf16 -> masked row stores; zero rows
//              that no group covers.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace gmm {

namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr uint64_t kDrainLimitNs = 200000000ull;

template <int BN, bool FUSE, bool BK>
struct Bf16Tile {
  // plain epilogue: rows staged in shared memory, one bulk copy per row
  static constexpr bool kStaged = !FUSE;
  static constexpr int kStages = (kStaged && BN == 256) ? 3 : 4;
  static constexpr int kStageRow = BN + 16;
  static constexpr int kStagingBytes = kStaged ? 2 * kBM * kStageRow : 0;
  static constexpr int kABytes = kBM * 64 * 2;   // 16 KB
  static constexpr int kBBytes = 64 * BN * 2;    // BN/64 boxes of 8 KB
  static constexpr int kBoxBytes = 64 * 64 * 2;  // one 64 x 64 bf16 box
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kOutCols = FUSE ? BN / 2 : BN;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + 256;
};

template <int BN, bool FUSE, bool BK>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_bf16_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const FwdArgs args) {
  static_assert(!(FUSE && BK), "the fused activation applies to the forward only");
  using C = Bf16Tile<BN, FUSE, BK>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  uint8_t* staging = smem + kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + C::kStagingBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_word = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_word = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();  // inputs and metadata come from earlier kernels

  const int num_tiles = args.meta[kWsNumTiles];
  const int units_per_tile = args.N / C::kOutCols;
  const long long num_units = static_cast<long long>(num_tiles) * units_per_tile;
  const int KS = args.K / 64;  // stages per unit
  const uint64_t lim = args.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t c = 0;
      bool ok = true;
      for (long long u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const Tile tl = args.tiles[u / units_per_tile];
        const int n0 = static_cast<int>(u % units_per_tile) * C::kOutCols;
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t s = c % kStages, ph = (c / kStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_word, lim)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = ring + s * C::kStageBytes;
          uint8_t* b_dst = a_dst + C::kABytes;
          mbar_arrive_expect_tx(&full[s], C::kStageBytes);
          tma_load_2d(a_dst, &map_a, &full[s], ks * 64, tl.row0);
          if (BK) {
            // K-major weight view [G*N_out, K]: BN rows of output columns
            tma_load_2d(b_dst, &map_b, &full[s], ks * 64, tl.g * args.N + n0);
          } else {
            const int wrow = tl.g * args.K + ks * 64;  // row of the [G*K, Nw] weight view
#pragma unroll
            for (int i = 0; i < BN / 64; ++i) {
              int col;
              if (FUSE) col = (i < BN / 128) ? n0 + 64 * i : args.N + n0 + 64 * (i - BN / 128);
              else col = n0 + 64 * i;
              tma_load_2d(b_dst + i * C::kBoxBytes, &map_b, &full[s], col, wrow);
            }
          }
          ++c;
        }
      }
      volatile int no_abort = 0;
      for (uint32_t s = 0; s < kStages; ++s) {
        if (c > s) {
          const uint32_t last = s + kStages * ((c - 1 - s) / kStages);
          mbar_wait(&full[s], (last / kStages) & 1u, &no_abort, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(1u /*bf16*/, false, !BK, kBM, BN);
      uint32_t c = 0, t = 0;
      bool ok = true;
      for (long long u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const uint32_t b = t & 1u, tph = (t >> 1) & 1u;
        if (!mbar_wait(&tempty[b], tph ^ 1u, abort_word, lim)) break;
        tc_fence_after();
        const uint32_t d = tbase + b * BN;
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t s = c % kStages, ph = (c / kStages) & 1u;
          if (!mbar_wait(&full[s], ph, abort_word, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(ring + s * C::kStageBytes);
          const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t bdesc = BK ? smem_desc_sw128(b_addr + 32 * j, 16, 1024)
                                      : smem_desc_sw128(b_addr + 2048 * j, C::kBoxBytes, 1024);
            mma_bf16(d, smem_desc_sw128(a_addr + 32 * j, 16, 1024), bdesc, idesc, (ks > 0 || j > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          ++c;
        }
        if (!ok) break;
        mma_commit(&tfull[b]);
        ++t;
      }
      if (c > 0) {
        volatile int no_abort = 0;
        mma_commit(drain);
        mbar_wait(drain, 0, &no_abort, kDrainLimitNs);
      }
    }
  } else {
    const int pw = warp - 2;
    const int h = pw >> 2;
    const int quad = warp & 3;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    {
      const int S = args.meta[kWsS];
      if (S < args.M) {
        const long long total = static_cast<long long>(args.M - S) * args.N / 8;
        uint4* p = reinterpret_cast<uint4*>(args.out + static_cast<long long>(S) * args.N);
        const long long stride = static_cast<long long>(gridDim.x) * (kEpiWarps * 32);
        for (long long i = static_cast<long long>(blockIdx.x) * (kEpiWarps * 32) + (threadIdx.x - 64); i < total;
             i += stride)
          p[i] = make_uint4(0, 0, 0, 0);
      }
    }
    uint32_t t = 0;
    for (long long u = blockIdx.x; u < num_units; u += gridDim.x) {
      const Tile tl = args.tiles[u / units_per_tile];
      const int n0 = static_cast<int>(u % units_per_tile) * C::kOutCols;
      const int row = tl.row0 + quad * 32 + lane;
      const bool valid = row < tl.row1;
      const uint32_t b = t & 1u, tph = (t >> 1) & 1u;
      const bool got = mbar_wait(&tfull[b], tph, abort_word, lim);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t tb = t_lane + b * BN;
      uint16_t* orow = args.out + static_cast<long long>(valid ? row : 0) * args.N;
      if (FUSE) {
        // gate columns [h*64, h*64+64), up columns BN/2 + the same
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t rg[32], ru[32];
          tmem_ld_32x32(tb + h * 64 + 32 * cc, rg);
          tmem_ld_32x32(tb + BN / 2 + h * 64 + 32 * cc, ru);
          tmem_ld_wait();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + n0 + h * 64 + 32 * cc);
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              float v[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) v[i] = silu_f32(__uint_as_float(rg[j + i])) * __uint_as_float(ru[j + i]);
              dst[j / 8] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                      pack_bf16x2(v[6], v[7]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
      } else {
        uint32_t r[BN / 2];
#pragma unroll
        for (int cc = 0; cc < BN / 64; ++cc)
          tmem_ld_32x32(tb + h * (BN / 2) + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * cc));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
        if (valid) {
          uint8_t* srow = staging + (h * kBM + quad * 32 + lane) * C::kStageRow;
          bulk_wait_read_all();
#pragma unroll
          for (int j = 0; j < BN / 2; j += 8) {
            reinterpret_cast<uint4*>(srow)[j / 8] =
                make_uint4(pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                           pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])),
                           pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5])),
                           pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7])));
          }
          fence_proxy_async_smem();
          bulk_copy_s2g(orow + n0 + h * (BN / 2), srow, BN);
          bulk_commit();
        }
      }
      ++t;
    }
    if (C::kStaged) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_word) atomicOr(const_cast<int32_t*>(args.meta) + kWsStatus, kErrTimeout);
}

template <int BN, bool FUSE, bool BK>
cudaError_t launch(const CUtensorMap& map_a, const CUtensorMap& map_b, const FwdArgs& args, int grid,
                   cudaStream_t stream) {
  constexpr int smem = Bf16Tile<BN, FUSE, BK>::kSmemBytes;
  cudaError_t e =
      cudaFuncSetAttribute(gmm_bf16_kernel<BN, FUSE, BK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(gmm_bf16_kernel<BN, FUSE, BK>, dim3(grid), dim3(kThreads), smem, stream, map_a, map_b, args);
}

}  // namespace

Fp8Geometry bf16_geometry(int N, int fuse) {
  if (fuse) return {256, 128, 64};
  if (N % 256 == 0) return {256, 256, 64};
  return {128, 128, 64};
}

cudaError_t launch_gmm_bf16(const CUtensorMap& map_a, const CUtensorMap& map_b, const FwdArgs& args, int grid,
                            cudaStream_t stream) {
  if (args.fuse) return launch<256, true, false>(map_a, map_b, args, grid, stream);
  if (args.N % 256 == 0) return launch<256, false, false>(map_a, map_b, args, grid, stream);
  return launch<128, false, false>(map_a, map_b, args, grid, stream);
}

cudaError_t launch_gmm_bf16_dgrad(const CUtensorMap& map_a, const CUtensorMap& map_b, const FwdArgs& args, int grid,
                                  cudaStream_t stream) {
  if (args.N % 256 == 0) return launch<256, false, true>(map_a, map_b, args, grid, stream);
  return launch<128, false, true>(map_a, map_b, args, grid, stream);
}

}  // namespace gmm
