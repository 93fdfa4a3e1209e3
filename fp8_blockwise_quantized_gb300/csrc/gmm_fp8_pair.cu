// a4-a6 on CTA pairs: the FP8 blockwise grouped GEMM forward with the
// 256-row MMA of two SMs (tcgen05 cta_group::2).
//
// Same arithmetic as gmm_fp8.cu ("GEMM Kernel 性能优化十问", Q1/Q3; "实现差距：
// GMM Kernel（V1 vs V2）", §3.3 and §3.5): for every 128-wide K block kb the
// exact FP8 partial P_kb is formed in fp32 on the tensor core and promoted with
// the LHS row scale times the RHS block scale, acc += P_kb * xs[kb, m] *
// ws[g, kb, n/128], in the same order, so the two kernels give the same bits.
//
// Why pairs.  With one CTA per tile the MMA of a 128x256 K block fills half of
// TMEM, so only two partials fit and the MMA of K block k+2 waits until the
// promotion warps have read the whole partial of K block k (two rounds of TMEM
// loads, the register file cannot hold a 128x256 partial next to the
// accumulators): the pipe drains once per K block.  Here a pair of CTAs owns a
// 256-row tile (128 rows each) and each K block is two M=256, N=128 MMAs
// ("halves") into four 128-column TMEM buffers: every promotion warp frees a
// half after one round of TMEM loads, and the MMA runs up to four halves ahead.
// The weight tile is split between the two CTAs (each loads 64 of a half's 128
// columns), so each SM's shared memory and L2 traffic per MMA stays what it
// is with one CTA and N = 256.  The price is the tile granularity: a group is
// cut into 256-row tiles, so a ragged group's last tile computes more rows
// that are not stored.
//
// Work unit = (256-row tile of one group, 256 weight columns): for the fused
// gate/up weight, half 0 is 128 gate columns and half 1 the 128 up columns of
// the same 128 output columns; otherwise the halves are output columns
// [n0, n0+128) and [n0+128, n0+256).  Per CTA (384 threads):
//   warp 0      TMA producer: per K block this CTA's 128x128 B Xq tile and its
//               64 columns of each half of the Wq tile (K-major, 128-byte
//               swizzle), 32 KB per stage.  The even CTA's full[s] takes both
//               CTAs' arrivals and bytes (the odd CTA's copies complete on it).
//   warp 1      even CTA: issues the MMAs (kind::f8f6f4, M=256, N=128, K=32,
//               four per half); commits arrive on both CTAs' barriers.
//   warp 2      scale loader (this CTA's 128 row scales + 2 block scales).
//   warp 3      store warp (staged bf16 boxes -> TMA / masked stores; the FP8
//               cast of h for the quantized output).
//   warps 4-11  promotion: warp (quadrant q, column group c) holds rows
//               32q..32q+31 and columns 64c..64c+63 of both halves (128 fp32
//               per thread); each half is one round of two TMEM loads, after
//               which the warp frees that buffer on the even CTA.
// Every wait is bounded; the pair leaves together through a cluster barrier.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tilewalk.cuh"

namespace gmm {

namespace {

constexpr int kThreads = 384;
constexpr int kPromoWarps = 8;
constexpr int kPromoWarp0 = 4;
constexpr uint32_t kRegControl = 56;
constexpr uint32_t kRegPromo = 224;
static_assert(128 * kRegControl + 256 * kRegPromo <= 384 * 168, "register split exceeds the launch budget");
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr int kScaleSlots = 8;
constexpr int kScaleSlotFloats = 132;  // 128 row scales + 2 block scales (+ pad)
constexpr int kTBufs = 4;              // TMEM buffers of one half (128 columns) each
constexpr int kHalfCols = 128;

template <bool FUSE, int STAGES>
struct PairTile {
  static constexpr int kBoxes = FUSE ? 1 : 2;  // 32x64 bf16 staging boxes per promotion warp
  static constexpr int kStagingBytes = kPromoWarps * kBoxes * 4096;
  static constexpr int kStages = STAGES;       // ring slots (default 5 fused, 4 otherwise)
  static constexpr int kABytes = kBM * 128;        // this CTA's 128 rows x 128 K bytes
  static constexpr int kBHalfBytes = 64 * 128;     // this CTA's 64 columns of a half
  static constexpr int kStageBytes = kABytes + 2 * kBHalfBytes;
  static constexpr int kOutCols = FUSE ? 128 : 256;  // output columns per unit
  static constexpr int kScaleBytes = kScaleSlots * kScaleSlotFloats * 4;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + kScaleBytes + kBarBytes;
  static_assert(8 * (2 * kStages + 2 * kTBufs + 2 * kScaleSlots + 3) + 8 <= kBarBytes, "barrier area");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

template <bool FUSE, bool QUANT, int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gmm_fp8_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_out, const FwdArgs args) {
  static_assert(!QUANT || FUSE, "the quantized output is for the fused units");
  using C = PairTile<FUSE, STAGES>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  uint8_t* staging = smem + S * C::kStageBytes;
  float* scales = reinterpret_cast<float*>(staging + C::kStagingBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(scales) + C::kScaleBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + kTBufs;  // even CTA: both CTAs' promotion warps freed buffer b
  uint64_t* sfull = tempty + kTBufs;
  uint64_t* sempty = sfull + kScaleSlots;
  uint64_t* staged = sempty + kScaleSlots;
  uint64_t* sfree = staged + 1;
  uint64_t* drain = sfree + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_word = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);  // both CTAs' producers (used on the even CTA)
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kTBufs; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * kPromoWarps);
    }
    for (int q = 0; q < kScaleSlots; ++q) {
      mbar_init(&sfull[q], 32);
      mbar_init(&sempty[q], kPromoWarps);
    }
    mbar_init(staged, kPromoWarps);
    mbar_init(sfree, 1);
    mbar_init(drain, 1);
    *abort_word = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
    tma_prefetch_desc(&map_out);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTBufs * kHalfCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();  // inputs and metadata come from earlier kernels

  const int num_tiles = args.meta[kWsNumPairTiles];
  const int units_per_tile = args.N / C::kOutCols;
  const uint32_t num_units = static_cast<uint32_t>(num_tiles) * static_cast<uint32_t>(units_per_tile);
  const bool col_major = args.col_major != 0;
  const int KB = args.K / 128;
  const int Nw = FUSE ? 2 * args.N : args.N;
  const uint64_t lim = args.wait_limit_ns;
  const uint32_t first = cluster_id_x(), step = cluster_count_x();
  // columns of W (rows of the K-major Wq) of half j of the unit at output column n0
  auto half_col = [&](int n0, int j) { return FUSE ? (j == 0 ? n0 : args.N + n0) : n0 + kHalfCols * j; };

  if (warp < kPromoWarp0) regs_dec<kRegControl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);
      // bytes this CTA's copies count per stage (4-bit weights: their packed
      // size, half of the e4m3 operand's shared-memory footprint)
      const uint32_t stage_tx = C::kABytes + (args.b_fmt != 0 ? C::kBHalfBytes : 2 * C::kBHalfBytes);
      uint32_t c = 0;
      bool ok = true;
      for (TileWalk w(args.pair_tiles, units_per_tile, num_units, num_tiles, col_major, first, step); w.live() && ok;
           w.next()) {
        const Tile tl = w.cur;
        const int n0 = w.col0(C::kOutCols);
        const int arow = tl.row0 + kBM * static_cast<int>(rank);
        const int b0 = tl.g * Nw + half_col(n0, 0) + 64 * static_cast<int>(rank);
        const int b1 = tl.g * Nw + half_col(n0, 1) + 64 * static_cast<int>(rank);
        for (int kb = 0; kb < KB; ++kb) {
          const uint32_t s = c % S, ph = (c / S) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_word, lim)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = ring + s * C::kStageBytes;
          uint8_t* b_dst = a_dst + C::kABytes;
          if (leader) {
            mbar_arrive_expect_tx(&full[s], stage_tx);
            tma_load_2d(a_dst, &map_a, &full[s], kb * 128, arow);
            tma_load_2d(b_dst, &map_b, &full[s], kb * 128, b0);
            tma_load_2d(b_dst + C::kBHalfBytes, &map_b, &full[s], kb * 128, b1);
          } else {
            // completes on the even CTA's barrier; the bytes may land before
            // the expectation is registered (the count dips below zero
            // within the phase)
            const uint32_t bar = full0 + s * 8u;
            mbar_arrive_expect_tx_remote(bar, stage_tx);
            tma_load_2d_pair(a_dst, &map_a, bar, kb * 128, arow);
            tma_load_2d_pair(b_dst, &map_b, bar, kb * 128, b0);
            tma_load_2d_pair(b_dst + C::kBHalfBytes, &map_b, bar, kb * 128, b1);
          }
          ++c;
        }
      }
      // the even CTA waits for the last copies into every slot (both CTAs'
      // land on its barriers) before the pair passes the teardown barrier
      volatile int no_abort = 0;
      for (uint32_t s = 0; leader && s < static_cast<uint32_t>(S); ++s) {
        if (c > s) {
          const uint32_t last = s + S * ((c - 1 - s) / S);
          mbar_wait(&full[s], (last / S) & 1u, &no_abort, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      // A e4m3; B e4m3, or e2m1 for 4-bit weights (bits 10-12)
      const uint32_t idesc = (make_idesc(0u /*e4m3*/, false, false, 2 * kBM, kHalfCols) & ~(7u << 10)) |
                             (static_cast<uint32_t>(args.b_fmt) << 10);
      uint32_t c = 0, t = 0;
      bool ok = true;
      for (uint32_t u = first; u < num_units && ok; u += step) {
        for (int kb = 0; kb < KB && ok; ++kb) {
          const uint32_t s = c % S, ph = (c / S) & 1u;
          if (!mbar_wait(&full[s], ph, abort_word, lim)) {
            ok = false;
            break;
          }
          const uint32_t a_addr = smem_u32(ring + s * C::kStageBytes);
#pragma unroll 1
          for (int j = 0; j < 2; ++j) {
            const uint32_t b = t % kTBufs, tph = (t / kTBufs) & 1u;
            if (!mbar_wait(&tempty[b], tph ^ 1u, abort_word, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t b_addr = a_addr + C::kABytes + j * C::kBHalfBytes;
            const uint32_t d = tbase + b * kHalfCols;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8_pair(d, smem_desc_sw128(a_addr + 32 * kk, 16, 1024), smem_desc_sw128(b_addr + 32 * kk, 16, 1024),
                          idesc, kk > 0 ? 1u : 0u);
            mma_commit_pair(&tfull[b], 0x3);
            ++t;
          }
          if (!ok) break;
          mma_commit_pair(&empty[s], 0x3);
          ++c;
        }
      }
      if (c > 0 || t > 0) {
        volatile int no_abort = 0;
        mma_commit_pair(drain, 0x1);
        mbar_wait(drain, 0, &no_abort, kDrainLimitNs);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale loader
    const int NBw = Nw / 128;
    uint32_t q = 0;
    bool ok = true;
    for (TileWalk w(args.pair_tiles, units_per_tile, num_units, num_tiles, col_major, first, step); w.live() && ok;
         w.next()) {
      const Tile tl = w.cur;
      const int n0 = w.col0(C::kOutCols);
      const int arow = tl.row0 + kBM * static_cast<int>(rank);
      const int wb0 = half_col(n0, 0) / 128, wb1 = half_col(n0, 1) / 128;
      const float* ws_g = args.ws + static_cast<long long>(tl.g) * KB * NBw;
      for (int kb = 0; kb < KB; ++kb) {
        const uint32_t sl = q % kScaleSlots, ph = (q / kScaleSlots) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&sempty[sl], ph ^ 1u, abort_word, lim))) {
          ok = false;
          break;
        }
        float* slot = scales + sl * kScaleSlotFloats;
        const float* xs_kb = args.xs + static_cast<long long>(kb) * args.M;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = lane * 4 + j;
          if (arow + r < args.M) cp_async_4(slot + r, xs_kb + arow + r);
        }
        if (lane == 0) {
          cp_async_4(slot + 128, ws_g + kb * NBw + wb0);
          cp_async_4(slot + 129, ws_g + kb * NBw + wb1);
        }
        cp_async_mbar_arrive_noinc(&sfull[sl]);
        ++q;
      }
    }
    cp_async_wait_all();
  } else if (warp == 3) {
    // ------------------------------------------------------------ store warp
    uint32_t ue = 0;
    bool ok = true;
    for (TileWalk w(args.pair_tiles, units_per_tile, num_units, num_tiles, col_major, first, step); w.live() && ok;
         w.next()) {
      const Tile tl = w.cur;
      const int n0 = w.col0(C::kOutCols);
      const int row0 = tl.row0 + kBM * static_cast<int>(rank);  // this CTA's rows
      const int row1 = min(tl.row1, row0 + kBM);
      if (!__all_sync(0xffffffffu, mbar_wait(staged, ue & 1u, abort_word, lim))) {
        ok = false;
        break;
      }
      if (args.out) {
        // box (p, i) of promotion warp p: rows row0 + (p & 3) * 32.., columns
        // n0 + (p >> 2) * 64 + 128 i; chunk j of row r at j ^ (r & 7)
        if (lane < kPromoWarps * C::kBoxes) {
          const int p = lane / C::kBoxes, i = lane % C::kBoxes;
          const int wrow0 = row0 + (p & 3) * 32;
          if (row1 - wrow0 >= 32) {
            tma_store_2d(&map_out, staging + (p * C::kBoxes + i) * 4096, n0 + (p >> 2) * 64 + kHalfCols * i, wrow0);
            bulk_commit();
          }
        }
        // ragged boxes (the tile ends inside this CTA's rows): masked stores
#pragma unroll 1
        for (int p = 0; p < kPromoWarps; ++p) {
          const int wrow0 = row0 + (p & 3) * 32;
          const int nvalid = min(32, row1 - wrow0);
          if (nvalid > 0 && nvalid < 32) {
            const uint8_t* wbox = staging + p * C::kBoxes * 4096;
            const int col0 = n0 + (p >> 2) * 64;
#pragma unroll 1
            for (int i = 0; i < C::kBoxes; ++i) {
#pragma unroll 1
              for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + (lane >> 3), j = lane & 7;
                if (r < nvalid)
                  *reinterpret_cast<uint4*>(args.out + static_cast<long long>(wrow0 + r) * args.N + col0 +
                                            kHalfCols * i + 8 * j) =
                      *reinterpret_cast<const uint4*>(wbox + i * 4096 + r * 128 + ((j ^ (r & 7)) << 4));
              }
            }
          }
        }
      }
      if (QUANT) {
        // h's 1x128 block of row r is the unit's 128 columns: box (r >> 5)
        // holds columns 0-63, box 4 + (r >> 5) columns 64-127
        const int nrows = row1 - row0;
        for (int r = lane; r < nrows; r += 32) {
          const int rr = r & 31, sw = r & 7;
          const uint8_t* b0 = staging + (r >> 5) * 4096 + rr * 128;
          const uint8_t* b1 = b0 + 4 * 4096;
          float amax = 0.0f;
#pragma unroll 2
          for (int j = 0; j < 8; ++j) {
            const uint4 v0 = *reinterpret_cast<const uint4*>(b0 + ((j ^ sw) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4*>(b1 + ((j ^ sw) << 4));
            amax = fmaxf(amax, fmaxf(bf16x8_absmax(v0), bf16x8_absmax(v1)));
          }
          float sc, inv;
          e4m3_block_scale(amax, sc, inv);
          uint8_t* qrow = args.hq + static_cast<long long>(row0 + r) * args.N + n0;
#pragma unroll 2
          for (int j = 0; j < 8; j += 2) {
            const uint2 q0 = bf16x8_to_e4m3(*reinterpret_cast<const uint4*>(b0 + ((j ^ sw) << 4)), inv);
            const uint2 q1 = bf16x8_to_e4m3(*reinterpret_cast<const uint4*>(b0 + (((j + 1) ^ sw) << 4)), inv);
            const uint2 q2 = bf16x8_to_e4m3(*reinterpret_cast<const uint4*>(b1 + ((j ^ sw) << 4)), inv);
            const uint2 q3 = bf16x8_to_e4m3(*reinterpret_cast<const uint4*>(b1 + (((j + 1) ^ sw) << 4)), inv);
            *reinterpret_cast<uint4*>(qrow + 8 * j) = make_uint4(q0.x, q0.y, q1.x, q1.y);
            *reinterpret_cast<uint4*>(qrow + 64 + 8 * j) = make_uint4(q2.x, q2.y, q3.x, q3.y);
          }
          args.hs[static_cast<long long>(n0 / 128) * args.M + row0 + r] = sc;
        }
      }
      bulk_wait_read_all();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree);
      ++ue;
    }
    bulk_wait_all();
  } else if (warp >= kPromoWarp0) {
    // ------------------------------------------------------------ promotion + epilogue
    regs_inc<kRegPromo>();
    const int pw = warp - kPromoWarp0;
    const int cg = pw >> 2;      // column group: columns 64 cg .. 64 cg + 63 of each half
    const int quad = warp & 3;   // TMEM lane quadrant this warp may access
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);

    // rows [S, M) belong to no group: zero them (spread over the whole grid)
    {
      const int S0 = args.meta[kWsS];
      if (S0 < args.M) {
        const long long total = static_cast<long long>(args.M - S0) * args.N / 8;
        uint4* p = reinterpret_cast<uint4*>(args.out + static_cast<long long>(S0) * args.N);
        const long long stride = static_cast<long long>(gridDim.x) * (kPromoWarps * 32);
        const long long tid =
            static_cast<long long>(blockIdx.x) * (kPromoWarps * 32) + (threadIdx.x - kPromoWarp0 * 32);
        if (args.out)
          for (long long i = tid; i < total; i += stride) p[i] = make_uint4(0, 0, 0, 0);
        if (QUANT) {
          uint4* qz = reinterpret_cast<uint4*>(args.hq + static_cast<long long>(S0) * args.N);
          for (long long i = tid; i < total / 2; i += stride) qz[i] = make_uint4(0, 0, 0, 0);
          const long long rows = args.M - S0;
          for (long long i = tid; i < rows * (args.N / 128); i += stride)
            args.hs[(i / rows) * args.M + S0 + (i % rows)] = 0.0f;
        }
      }
    }

    uint32_t t = 0, q = 0, ue = 0;
    bool ok = true;
    for (TileWalk w(args.pair_tiles, units_per_tile, num_units, num_tiles, col_major, first, step); w.live() && ok;
         w.next()) {
      const Tile tl = w.cur;
      const int row0 = tl.row0 + kBM * static_cast<int>(rank);
      const int row1 = min(tl.row1, row0 + kBM);
      const int rit = quad * 32 + lane;  // row within this CTA's 128
      const bool valid = row0 + rit < row1;
      // acc[0..31]: half 0, columns 64 cg + 2i, 2i+1; acc[32..63]: half 1
      float2 acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);

      for (int kb = 0; kb < KB && ok; ++kb) {
        const uint32_t sl = q % kScaleSlots, sph = (q / kScaleSlots) & 1u;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t b = t % kTBufs, tph = (t / kTBufs) & 1u;
          bool got = mbar_wait(&tfull[b], tph, abort_word, lim);
          if (j == 0) got = got && mbar_wait(&sfull[sl], sph, abort_word, lim);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          const float* slot = scales + sl * kScaleSlotFloats;
          const float sx = valid ? slot[rit] : 0.0f;
          const float f = sx * slot[128 + j];
          tc_fence_after();
          uint32_t ra[32], rb[32];
          const uint32_t tb = t_lane + b * kHalfCols + 64 * cg;
          tmem_ld_32x32(tb, ra);
          tmem_ld_32x32(tb + 32, rb);
          tmem_ld_wait();
          // the half is in registers: hand its buffer back to the pair's MMA
          // issuer (and the scale slot after the second half)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_remote(tempty0 + b * 8u);
            if (j == 1) mbar_arrive(&sempty[sl]);
          }
          const float2 ff = make_float2(f, f);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[32 * j + i] =
                __ffma2_rn(make_float2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1])), ff, acc[32 * j + i]);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[32 * j + 16 + i] = __ffma2_rn(make_float2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1])),
                                              ff, acc[32 * j + 16 + i]);
          ++t;
        }
        ++q;
      }
      if (!ok) break;
      // epilogue: once the store warp has emptied the staging area, this
      // warp's 32 rows go in as bf16 boxes (chunk j of row r at j ^ (r & 7))
      if (!__all_sync(0xffffffffu, mbar_wait(sfree, (ue & 1u) ^ 1u, abort_word, lim))) break;
      uint8_t* wbox = staging + pw * C::kBoxes * 4096 + lane * 128;
      if (FUSE) {
        // h = bf16(silu(gate) * up): gate in half 0, up in half 1
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t hb[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 gt = acc[4 * j + k], up = acc[32 + 4 * j + k];
            hb[k] = pack_bf16x2(silu_f32(gt.x) * up.x, silu_f32(gt.y) * up.y);
          }
          *reinterpret_cast<uint4*>(wbox + ((j ^ (lane & 7)) << 4)) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int p2 = 32 * i + 4 * j;
            *reinterpret_cast<uint4*>(wbox + i * 4096 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(pack_bf16x2(acc[p2].x, acc[p2].y), pack_bf16x2(acc[p2 + 1].x, acc[p2 + 1].y),
                           pack_bf16x2(acc[p2 + 2].x, acc[p2 + 2].y), pack_bf16x2(acc[p2 + 3].x, acc[p2 + 3].y));
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(staged);
      ++ue;
    }
  }

  // ------------------------------------------------------------ teardown
  // no CTA of the pair leaves while the other may still arrive on its
  // barriers or the pair's MMAs may still write its TMEM
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, kTBufs * kHalfCols);
  }
  if (threadIdx.x == 0 && *abort_word) atomicOr(const_cast<int32_t*>(args.meta) + kWsStatus, kErrTimeout);
}

template <bool FUSE, bool QUANT, int STAGES>
cudaError_t launch(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                   const FwdArgs& args, int max_pairs, cudaStream_t stream) {
  constexpr int smem = PairTile<FUSE, STAGES>::kSmemBytes;
  auto kernel = gmm_fp8_pair_kernel<FUSE, QUANT, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // as many pairs as can be resident at once (one CTA per SM)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * max_pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int pairs = clusters < max_pairs ? clusters : max_pairs;
  return launch_pdl(kernel, dim3(2 * pairs), dim3(kThreads), smem, stream, map_a, map_b, map_out, args);
}

template <bool FUSE, bool QUANT>
cudaError_t launch_stages(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                          const FwdArgs& args, int max_pairs, cudaStream_t stream) {
  if (args.stages == 3) return launch<FUSE, QUANT, 3>(map_a, map_b, map_out, args, max_pairs, stream);
  if constexpr (FUSE) {
    if (args.stages != 4) return launch<FUSE, QUANT, 5>(map_a, map_b, map_out, args, max_pairs, stream);
  }
  return launch<FUSE, QUANT, 4>(map_a, map_b, map_out, args, max_pairs, stream);
}

}  // namespace

cudaError_t launch_gmm_fp8_pair(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                                const FwdArgs& args, int max_pairs, cudaStream_t stream) {
  if (args.fuse && args.hq) return launch_stages<true, true>(map_a, map_b, map_out, args, max_pairs, stream);
  if (args.fuse) return launch_stages<true, false>(map_a, map_b, map_out, args, max_pairs, stream);
  return launch_stages<false, false>(map_a, map_b, map_out, args, max_pairs, stream);
}

}  // namespace gmm
