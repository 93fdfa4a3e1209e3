#pragma once
// a4-a6: FP8 blockwise grouped GEMM forward on the 5th-generation tensor core
// (the single-CTA kernel template; instantiated by gmm_fp8.cu and gmm_fp8_n128.cu).
//
// What it computes ("GEMM Kernel 性能优化十问", Q1/Q3; "实现差距：GMM Kernel
// （V1 vs V2）", §3.3 and §3.5): for the row tile (g, row0..row1) and a column
// block, for every 128-wide K block kb (one LHS / RHS quantization block) the
// exact FP8 partial P_kb = Xq[rows, kb] . Wq[g][kb, cols] is formed in fp32 and
// promoted into the accumulator with the LHS row scale times the RHS block
// scale: acc += P_kb * xs[kb, m] * ws[g, kb, n/128].  The output is bf16(acc),
// or bf16(silu(acc_gate) * acc_up) with the fused gate/up weight.
//
// How (sm_103a).  The quantization block is decoupled from the pipeline: the
// MMA never stops at a block boundary, only its accumulator buffer changes.
//   warp 0      TMA producer: per K block one 128x128 B Xq tile and one
//               BNx128 B Wq tile (K-major, 128-byte swizzle) into a shared-
//               memory ring of STAGES slots (by default 3 of 48 KB with
//               BN = 256, 4 of 32 KB with BN = 128), completion counted on an
//               mbarrier.
//   warp 1      allocates TMEM and issues tcgen05.mma (kind::f8f6f4, M=128,
//               N=BN, K=32, four per K block) into one of NBUF TMEM partial
//               buffers (2; or 4 with BN = 128, all 512 columns);
//               tcgen05.commit frees the ring slot and publishes the partial.
//   warp 2      unit scheduler and scale loader: claims the CTA's next unit
//               from a counter in the workspace and hands it to the other
//               roles through a shared-memory queue; then, per K block,
//               cp.async copies of the tile's 128 row scales xs[kb, rows] and
//               its RHS block scales into a shared-memory ring that runs ahead
//               of the MMAs (the scales are then never a global-memory load on
//               the promotion's path).
//   warp 3      store warp: takes each unit's staged bf16 output boxes to
//               global memory (TMA tensor stores for full 32-row boxes, masked
//               stores for ragged ones: the tile may run into the next group)
//               and, for the quantized output, re-reads the staged bf16 rows
//               to cast them to e4m3 with 1x128 absmax scales.
//   warps 4-11  promotion: tcgen05.ld the partial (one TMEM lane = one row),
//               FMA it into fp32 registers with the scale product, release the
//               buffer; after the last K block convert the accumulators to
//               bf16 (silu(gate) * up when fused) into swizzled 32x64 staging
//               boxes and go on with the next unit while the store warp
//               drains them.  They also zero the output rows no group covers.
// Work units (tile, column block) are claimed by a persistent grid of one CTA
// per SM from a counter as the CTAs go (list scheduling: a CTA that runs
// slower takes fewer), numbered tile-major so that the units sharing an Xq
// tile and the tiles sharing an expert's Wq columns run at the same time (L2
// reuse).  The last CTA to finish resets the counter for the next launch.
// Every wait is bounded; a timeout sets the workspace error word and all
// roles unwind, wait for their copies and MMAs in flight and free TMEM.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace gmm {

namespace {

constexpr int kThreads = 384;
constexpr int kPromoWarps = 8;
constexpr int kPromoWarp0 = 4;   // first promotion warp
// Register split: the launch gives 168 registers per thread (three warps per
// SM sub-partition); warpgroup 0 (TMA, MMA, scales, stores) gives most of its
// share to the two promotion warpgroups, which hold the fp32 accumulators:
// 128 x control + 256 x promo <= 384 x 168 = 64512.
template <int BN>
struct RegSplit {
  static constexpr uint32_t kControl = BN == 256 ? 56 : 72;
  static constexpr uint32_t kPromo = BN == 256 ? 224 : 216;
  static_assert(128 * kControl + 256 * kPromo <= 384 * 168, "register split exceeds the launch budget");
};
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr int kScaleSlots = 8;        // K blocks of scales in flight
constexpr int kUnitSlots = 8;         // entries of the CTA's unit queue
// readers of a queue entry: producer, MMA issuer, store warp, promotion warps
constexpr int kUnitReaders = 3 + 8;

// The CTA's unit queue: the scale loader claims each unit from a counter in
// the workspace and writes {g, row0, row1, first output column} (g < 0: no
// more units) to entry i % kUnitSlots; every other role takes the entries in
// order and frees each one it has read.
struct FwdUnitQueue {
  uint64_t* full;
  uint64_t* empty;
  const int4* data;
  __device__ bool get(uint32_t i, int4& e, bool warp_wide, int lane, volatile int* abort_word, uint64_t lim) const {
    const uint32_t slot = i % kUnitSlots, ph = (i / kUnitSlots) & 1u;
    bool ok = mbar_wait(&full[slot], ph, abort_word, lim);
    if (warp_wide) ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    e = data[slot];
    if (warp_wide) __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    return true;
  }
};
constexpr int kScaleSlotFloats = 132;  // 128 row scales + 2 block scales (+ pad)

template <int BN, bool FUSE, bool QUANT, int STAGES, int NBUF>
struct Fp8Tile {
  // The epilogue stages each promotion warp's 32 output rows as bf16 boxes of
  // 32 rows x 64 columns (4 KB, 128-byte swizzle): BN/128 boxes per warp, or
  // one box of h when fused.  STAGES ring slots (default 3 with BN = 256,
  // the staging taking the room of a fourth; 4 with BN = 128).
  static constexpr int kStages = STAGES;
  static constexpr int kBoxes = FUSE ? 1 : BN / 128;
  static constexpr int kStagingBytes = 8 * kBoxes * 4096;
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kSeg = BN / 4;                  // columns per accumulator segment
  static constexpr int kOutCols = FUSE ? BN / 2 : BN;  // output columns per work unit
  static constexpr int kBufs = NBUF;                   // TMEM partial buffers (2, or 4 with BN = 128)
  static constexpr int kTmemCols = NBUF * BN;
  static_assert(kTmemCols <= 512, "TMEM holds 512 columns");
  static constexpr int kBarBytes = 768;  // barriers, then the unit queue's entries
  static constexpr int kScaleBytes = kScaleSlots * kScaleSlotFloats * 4;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + kScaleBytes + kBarBytes;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(8 * (2 * kStages + 2 * NBUF + 2 * kScaleSlots + 3 + 2 * kUnitSlots) + 32 + 16 * kUnitSlots <=
                    kBarBytes,
                "barrier area");
};

template <int BN, bool FUSE, bool QUANT, int STAGES, int NBUF>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_fp8_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_out, const FwdArgs args) {
  static_assert(!QUANT || (FUSE && BN == 256), "the quantized output is for the fused 128-column units");
  using C = Fp8Tile<BN, FUSE, QUANT, STAGES, NBUF>;
  constexpr int SEG = C::kSeg;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  uint8_t* staging = smem + kStages * C::kStageBytes;
  float* scales = reinterpret_cast<float*>(staging + C::kStagingBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(scales) + C::kScaleBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + NBUF;
  uint64_t* sfull = tempty + NBUF;
  uint64_t* sempty = sfull + kScaleSlots;
  uint64_t* staged = sempty + kScaleSlots;  // a unit's output boxes are in the staging area
  uint64_t* sfree = staged + 1;             // the store warp has emptied the staging area
  uint64_t* drain = sfree + 1;
  uint64_t* ufull = drain + 1;          // unit queue entry written
  uint64_t* uempty = ufull + kUnitSlots;  // unit queue entry read by every reader
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(uempty + kUnitSlots);
  volatile int* abort_word = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int4* udata = reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(tmem_slot + 2) + 15) & ~uintptr_t{15});

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kPromoWarps);
    }
    for (int q = 0; q < kScaleSlots; ++q) {
      mbar_init(&sfull[q], 32);  // one cp.async arrival per loader lane
      mbar_init(&sempty[q], kPromoWarps);
    }
    mbar_init(staged, kPromoWarps);
    mbar_init(sfree, 1);
    mbar_init(drain, 1);
    for (int q = 0; q < kUnitSlots; ++q) {
      mbar_init(&ufull[q], 1);
      mbar_init(&uempty[q], kUnitReaders);
    }
    *abort_word = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
    tma_prefetch_desc(&map_out);
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
  const uint32_t num_units = static_cast<uint32_t>(num_tiles) * static_cast<uint32_t>(units_per_tile);
  const bool col_major = args.col_major != 0;
  const int KB = args.K / 128;
  const int Nw = FUSE ? 2 * args.N : args.N;
  const uint64_t lim = args.wait_limit_ns;
  const FwdUnitQueue queue{ufull, uempty, udata};

  if (warp < kPromoWarp0) regs_dec<RegSplit<BN>::kControl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // bytes a stage's copies count on its barrier: 4-bit weights count
      // their packed size (64 bytes per 128-code row), though they land
      // expanded to the e4m3 operand's footprint in shared memory
      const uint32_t stage_tx = C::kABytes + (args.b_fmt != 0 ? C::kBBytes / 2 : C::kBBytes);
      uint32_t c = 0;
      bool ok = true;
      int4 e;
      for (uint32_t i = 0; ok && queue.get(i, e, false, 0, abort_word, lim) && e.x >= 0; ++i) {
        const Tile tl{e.x, e.y, e.z, 0};
        const int n0 = e.w;
        const int brow = tl.g * Nw + n0;
        for (int kb = 0; kb < KB; ++kb) {
          const uint32_t s = c % kStages, ph = (c / kStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_word, lim)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = ring + s * C::kStageBytes;
          uint8_t* b_dst = a_dst + C::kABytes;
          mbar_arrive_expect_tx(&full[s], stage_tx);
          tma_load_2d(a_dst, &map_a, &full[s], kb * 128, tl.row0);
          if (FUSE) {
            tma_load_2d(b_dst, &map_b, &full[s], kb * 128, brow);
            tma_load_2d(b_dst + C::kBBytes / 2, &map_b, &full[s], kb * 128, brow + args.N);
          } else {
            tma_load_2d(b_dst, &map_b, &full[s], kb * 128, brow);
          }
          ++c;
        }
      }
      // wait for the last copy issued into every slot (they land in microseconds)
      volatile int no_abort = 0;
      for (uint32_t s = 0; s < kStages; ++s) {
        if (c > s) {
          const uint32_t last = s + kStages * ((c - 1 - s) / kStages);
          mbar_wait(&full[s], (last / kStages) & 1u, &no_abort, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // A e4m3; B e4m3, or e2m1 for 4-bit weights (bits 10-12)
      const uint32_t idesc =
          (make_idesc(0u /*e4m3*/, false, false, kBM, BN) & ~(7u << 10)) | (static_cast<uint32_t>(args.b_fmt) << 10);
      uint32_t c = 0, t = 0;
      bool ok = true;
      int4 e;
      for (uint32_t i = 0; ok && queue.get(i, e, false, 0, abort_word, lim) && e.x >= 0; ++i) {
        for (int kb = 0; kb < KB; ++kb) {
          const uint32_t s = c % kStages, ph = (c / kStages) & 1u;
          if (!mbar_wait(&full[s], ph, abort_word, lim)) {
            ok = false;
            break;
          }
          const uint32_t b = t % NBUF, tph = (t / NBUF) & 1u;
          if (!mbar_wait(&tempty[b], tph ^ 1u, abort_word, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(ring + s * C::kStageBytes);
          const uint32_t b_addr = a_addr + C::kABytes;
          const uint32_t d = tbase + b * BN;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            mma_f8(d, smem_desc_sw128(a_addr + 32 * j, 16, 1024), smem_desc_sw128(b_addr + 32 * j, 16, 1024),
                   idesc, j > 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          mma_commit(&tfull[b]);
          ++c;
          ++t;
        }
      }
      if (c > 0) {
        volatile int no_abort = 0;
        mma_commit(drain);
        mbar_wait(drain, 0, &no_abort, kDrainLimitNs);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ unit scheduler and scale loader
    // Claims units from the workspace counter (units u = row tile u / per_tile,
    // column block u % per_tile, or column-block major), one claim in flight
    // while the current unit is published and its scales are loaded.
    const int NBw = Nw / 128;
    int* claimed = const_cast<int32_t*>(args.meta) + kWsClaimed;
    uint32_t q = 0;
    bool ok = true;
    int mine = 0;
    if (lane == 0) mine = atomicAdd(claimed, 1);
    for (uint32_t i = 0; ok; ++i) {
      const int u = __shfl_sync(0xffffffffu, mine, 0);
      const bool live = u < static_cast<int>(num_units);
      if (live && lane == 0) mine = atomicAdd(claimed, 1);
      int4 ent = make_int4(-1, 0, 0, 0);
      if (live) {
        const uint32_t tix = col_major ? static_cast<uint32_t>(u) % static_cast<uint32_t>(num_tiles)
                                       : static_cast<uint32_t>(u) / static_cast<uint32_t>(units_per_tile);
        const int col = col_major ? u / num_tiles : u % units_per_tile;
        const int4 t = __ldg(reinterpret_cast<const int4*>(args.tiles + tix));
        ent = make_int4(t.x, t.y, t.z, col * C::kOutCols);
      }
      {
        const uint32_t slot = i % kUnitSlots, ph = (i / kUnitSlots) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&uempty[slot], ph ^ 1u, abort_word, lim))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          udata[slot] = ent;
          mbar_arrive(&ufull[slot]);
        }
        __syncwarp();
      }
      if (!live) break;
      const Tile tl{ent.x, ent.y, ent.z, 0};
      const int n0 = ent.w;
      // the (up to) two RHS column blocks this unit's accumulators use
      const int wb0 = n0 / 128;
      const int wb1 = FUSE ? (args.N + n0) / 128 : (BN == 256 ? n0 / 128 + 1 : n0 / 128);
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
          if (tl.row0 + r < args.M) cp_async_4(slot + r, xs_kb + tl.row0 + r);
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
    int4 e;
    for (uint32_t i = 0; ok && queue.get(i, e, true, lane, abort_word, lim) && e.x >= 0; ++i) {
      const Tile tl{e.x, e.y, e.z, 0};
      const int n0 = e.w;
      if (!__all_sync(0xffffffffu, mbar_wait(staged, ue & 1u, abort_word, lim))) {
        ok = false;
        break;
      }
      if (args.out) {
        // box region of promotion warp p: rows (p & 3) * 32.., columns
        // n0 + (p >> 2) * 64 * kBoxes..; chunk j of row r at j ^ (r & 7).
        // Full 32-row boxes: one TMA tensor store per box, issued by lanes
        // in parallel (lane = p * kBoxes + box).
        if (lane < kPromoWarps * C::kBoxes) {
          const int p = lane / C::kBoxes, i = lane % C::kBoxes;
          const int wrow0 = tl.row0 + (p & 3) * 32;
          if (tl.row1 - wrow0 >= 32) {
            tma_store_2d(&map_out, staging + (p * C::kBoxes + i) * 4096, n0 + (p >> 2) * 64 * C::kBoxes + 64 * i,
                         wrow0);
            bulk_commit();
          }
        }
        // ragged boxes (the tile runs into the next group): masked stores
#pragma unroll 1
        for (int p = 0; p < kPromoWarps; ++p) {
          const int wrow0 = tl.row0 + (p & 3) * 32;
          const int nvalid = min(32, tl.row1 - wrow0);
          if (nvalid > 0 && nvalid < 32) {
            const uint8_t* wbox = staging + p * C::kBoxes * 4096;
            const int col0 = n0 + (p >> 2) * 64 * C::kBoxes;
#pragma unroll 1
            for (int i = 0; i < C::kBoxes; ++i) {
#pragma unroll 1
              for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + (lane >> 3), j = lane & 7;
                if (r < nvalid)
                  *reinterpret_cast<uint4*>(args.out + static_cast<long long>(wrow0 + r) * args.N + col0 + 64 * i +
                                            8 * j) =
                      *reinterpret_cast<const uint4*>(wbox + i * 4096 + r * 128 + ((j ^ (r & 7)) << 4));
              }
            }
          }
        }
      }
      if (QUANT) {
        // h's 1x128 block of row r is the unit's 128 columns: box (r >> 5)
        // holds columns 0-63, box 4 + (r >> 5) columns 64-127.  Quantized
        // exactly as gmm_quantize_lhs would: absmax of the bf16 values / 448.
        const int nrows = tl.row1 - tl.row0;
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
          uint8_t* qrow = args.hq + static_cast<long long>(tl.row0 + r) * args.N + n0;
#pragma unroll 2
          for (int j = 0; j < 8; j += 2) {
            const uint2 q0 = bf16x8_to_e4m3(*reinterpret_cast<const uint4*>(b0 + ((j ^ sw) << 4)), inv);
            const uint2 q1 = bf16x8_to_e4m3(*reinterpret_cast<const uint4*>(b0 + (((j + 1) ^ sw) << 4)), inv);
            const uint2 q2 = bf16x8_to_e4m3(*reinterpret_cast<const uint4*>(b1 + ((j ^ sw) << 4)), inv);
            const uint2 q3 = bf16x8_to_e4m3(*reinterpret_cast<const uint4*>(b1 + (((j + 1) ^ sw) << 4)), inv);
            *reinterpret_cast<uint4*>(qrow + 8 * j) = make_uint4(q0.x, q0.y, q1.x, q1.y);
            *reinterpret_cast<uint4*>(qrow + 64 + 8 * j) = make_uint4(q2.x, q2.y, q3.x, q3.y);
          }
          args.hs[static_cast<long long>(n0 / 128) * args.M + tl.row0 + r] = sc;
        }
      }
      // the staging area may be overwritten once the tensor stores have read
      // it (each issuing lane waits for its own) and every lane's reads are done
      bulk_wait_read_all();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree);
      ++ue;
    }
    bulk_wait_all();
  } else if (warp >= kPromoWarp0) {
    // ------------------------------------------------------------ promotion + epilogue
    regs_inc<RegSplit<BN>::kPromo>();
    const int pw = warp - kPromoWarp0;
    const int h = pw >> 2;        // column half of the tile
    const int quad = warp & 3;    // TMEM lane quadrant this warp may access
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quad * 32) << 16);

    // rows [S, M) belong to no group: zero them (spread over the whole grid)
    {
      const int S = args.meta[kWsS];
      if (S < args.M) {
        const long long total = static_cast<long long>(args.M - S) * args.N / 8;
        uint4* p = reinterpret_cast<uint4*>(args.out + static_cast<long long>(S) * args.N);
        const long long stride = static_cast<long long>(gridDim.x) * (kPromoWarps * 32);
        const long long tid = static_cast<long long>(blockIdx.x) * (kPromoWarps * 32) + (threadIdx.x - kPromoWarp0 * 32);
        if (args.out)
          for (long long i = tid; i < total; i += stride) p[i] = make_uint4(0, 0, 0, 0);
        if (QUANT) {
          // codes 0 and scale 0, as quantizing the zero rows gives
          uint4* q = reinterpret_cast<uint4*>(args.hq + static_cast<long long>(S) * args.N);
          for (long long i = tid; i < total / 2; i += stride) q[i] = make_uint4(0, 0, 0, 0);
          const long long rows = args.M - S;
          for (long long i = tid; i < rows * (args.N / 128); i += stride)
            args.hs[(i / rows) * args.M + S + (i % rows)] = 0.0f;
        }
      }
    }

    uint32_t t = 0, ue = 0;
    bool ok = true;
    int4 e;
    for (uint32_t i = 0; ok && queue.get(i, e, true, lane, abort_word, lim) && e.x >= 0; ++i) {
      const Tile tl{e.x, e.y, e.z, 0};
      const int row = tl.row0 + quad * 32 + lane;
      const bool valid = row < tl.row1;
      int tcol0, tcol1, wsel0, wsel1;
      if (FUSE) {
        tcol0 = h * SEG;
        tcol1 = BN / 2 + h * SEG;
        wsel0 = 0;  // gate block
        wsel1 = 1;  // up block
      } else {
        tcol0 = h * (BN / 2);
        tcol1 = h * (BN / 2) + SEG;
        wsel0 = wsel1 = (BN == 256) ? h : 0;
      }
      const int rit = quad * 32 + lane;  // row within the tile
      // fp32 accumulators, kept as pairs for the packed FMA: acc[2i], acc[2i+1]
      float2 acc[SEG];
#pragma unroll
      for (int i = 0; i < SEG; ++i) acc[i] = make_float2(0.0f, 0.0f);

      for (int kb = 0; kb < KB; ++kb) {
        const uint32_t b = t % NBUF, tph = (t / NBUF) & 1u;
        const uint32_t sl = t % kScaleSlots, sph = (t / kScaleSlots) & 1u;
        const bool got = mbar_wait(&tfull[b], tph, abort_word, lim) && mbar_wait(&sfull[sl], sph, abort_word, lim);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const float* slot = scales + sl * kScaleSlotFloats;
        const float sx = valid ? slot[rit] : 0.0f;
        const float sw0 = slot[128 + wsel0], sw1 = slot[128 + wsel1];
        tc_fence_after();
        const float f0 = sx * sw0, f1 = sx * sw1;
        const uint32_t tb = t_lane + b * BN;
        // 32-column chunks: the first SEG/32 belong to segment 0, the rest to
        // segment 1.  Two TMEM loads are in flight per wait.
        constexpr int NCH = 2 * SEG / 32, CPS = SEG / 32;
#pragma unroll
        for (int pc = 0; pc < NCH; pc += 2) {
          uint32_t ra[32], rb[32];
          const int ca = pc, cb = pc + 1;
          tmem_ld_32x32(tb + (ca < CPS ? tcol0 + 32 * ca : tcol1 + 32 * (ca - CPS)), ra);
          tmem_ld_32x32(tb + (cb < CPS ? tcol0 + 32 * cb : tcol1 + 32 * (cb - CPS)), rb);
          tmem_ld_wait();
          if (pc == NCH - 2) {
            // the K block's partial is in registers: hand the buffer and the
            // scale slot back before the last multiply-adds
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&tempty[b]);
              mbar_arrive(&sempty[sl]);
            }
          }
          const float2 fa = ca < CPS ? make_float2(f0, f0) : make_float2(f1, f1);
          const float2 fb = cb < CPS ? make_float2(f0, f0) : make_float2(f1, f1);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[16 * ca + i] =
                __ffma2_rn(make_float2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1])), fa,
                           acc[16 * ca + i]);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[16 * cb + i] =
                __ffma2_rn(make_float2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1])), fb,
                           acc[16 * cb + i]);
        }
        ++t;
      }
      if (!ok) break;
      // epilogue: once the store warp has emptied the staging area, this
      // warp's 32 rows go in as bf16 boxes (chunk j of row r at j ^ (r & 7))
      if (!__all_sync(0xffffffffu, mbar_wait(sfree, (ue & 1u) ^ 1u, abort_word, lim))) break;
      uint8_t* wbox = staging + pw * C::kBoxes * 4096 + lane * 128;
      if (FUSE) {
        // gate = acc[0, SEG/2), up = acc[SEG/2, SEG) (pairs of columns);
        // h = bf16(silu(gate) * up), SEG = 64 columns = one box row
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t hb[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 gt = acc[4 * j + k], up = acc[SEG / 2 + 4 * j + k];
            hb[k] = pack_bf16x2(silu_f32(gt.x) * up.x, silu_f32(gt.y) * up.y);
          }
          *reinterpret_cast<uint4*>(wbox + ((j ^ (lane & 7)) << 4)) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < C::kBoxes; ++i) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int p2 = 32 * i + 4 * j;  // float2 index of column 64 i + 8 j
            *reinterpret_cast<uint4*>(wbox + i * 4096 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(pack_bf16x2(acc[p2].x, acc[p2].y), pack_bf16x2(acc[p2 + 1].x, acc[p2 + 1].y),
                           pack_bf16x2(acc[p2 + 2].x, acc[p2 + 2].y), pack_bf16x2(acc[p2 + 3].x, acc[p2 + 3].y));
          }
        }
      }
      fence_proxy_async_smem();  // the tensor stores read the boxes through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(staged);
      ++ue;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
  if (threadIdx.x == 0) {
    int32_t* w = const_cast<int32_t*>(args.meta);
    if (*abort_word) atomicOr(w + kWsStatus, kErrTimeout);
    // every CTA has stopped claiming; the last one out resets the counters
    __threadfence();
    if (atomicAdd(w + kWsFinished, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(w + kWsClaimed, 0);
      atomicExch(w + kWsFinished, 0);
    }
  }
}

template <int BN, bool FUSE, bool QUANT, int STAGES, int NBUF>
cudaError_t launch(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_out,
                   const FwdArgs& args, int grid, cudaStream_t stream) {
  constexpr int smem = Fp8Tile<BN, FUSE, QUANT, STAGES, NBUF>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(gmm_fp8_kernel<BN, FUSE, QUANT, STAGES, NBUF>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(gmm_fp8_kernel<BN, FUSE, QUANT, STAGES, NBUF>, dim3(grid), dim3(kThreads), smem, stream, map_a,
                    map_b, map_out, args);
}

}  // namespace

}  // namespace gmm
