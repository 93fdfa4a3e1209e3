// a8: tgmm, the expert weight gradient in bf16.
//
// dW[g][k, n] = sum over the rows m of group g of x[m, k] * dy[m, n]
// ("GEMM Kernel 性能优化十问", Q4: dW[K,N] += X^T[K,M] dY[M,N], M is the
// reduction dimension; Q5: the backward pass is not quantized).  fp32
// accumulation, bf16 output; an empty group gets dW[g] = 0.
//
// Work unit = one output tile (g, 128 rows of K, BN columns of N).  Its
// reduction walks the group's rows in chunks of 64:
//   warp 0     TMA: x[rows, 128 k] as two 64x64 boxes and dy[rows, BN n] as
//              BN/64 boxes; both land MN-major (K of the MMA = the row index).
//   warp 1     tcgen05.mma kind::f16, M=128 (k), N=BN (n), K=16 (rows).  On
//              the group's last, partial chunk it skips the 16-row steps past
//              the group's end and zeroes the x rows of the last step that
//              belong to the next group (whole 128-byte rows, so the swizzle
//              does not matter), fenced into the async proxy.
//   warps 2-9  epilogue: tcgen05.ld -> bf16 -> the warp's 32 rows staged in
//              shared memory one 32x64 box at a time (128-byte swizzle) -> one
//              TMA tensor store per box; zero tile for an empty group.  The
//              small staging area leaves room for a 4-slot load ring.
// TMEM holds two accumulators, so one tile's epilogue overlaps the next
// tile's MMAs.  Units are numbered group-major, largest groups first, so the
// tiles of one group (which share its x and dy rows) run together; this
// single-CTA kernel (K not a multiple of 256) deals them in snake rounds, the
// CTA-pair kernel below claims them from a counter.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace gmm {

namespace {

constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kChunk = 64;  // rows per stage
constexpr uint64_t kDrainLimitNs = 200000000ull;

// The units of a launch are numbered group by group, the groups taken
// largest first (`order`: the groups by size, descending), and dealt to the
// CTAs (or CTA pairs) in snake order: round r gives unit r * stride + first
// when r is even and r * stride + stride - 1 - first when it is odd.  The big
// units come first and each CTA's rounds alternate ends, so the last wave
// holds small units and the loads stay balanced.  Unit u covers group
// order[u / per_group], column/row block u % per_group.  The next unit's group
// and offsets are loaded one unit ahead, so their global-memory latency
// overlaps the current unit.
struct UnitWalk {
  const int* offsets;
  const int* order;
  int per_group, num, step, first, round, u, g, rem, r0, r1, un, gn, r0n, r1n;
  __device__ int unit_of(int r) const { return r * step + ((r & 1) ? step - 1 - first : first); }
  __device__ UnitWalk(const int* off, const int* ord, int per_group_units, int num_units, int first_unit,
                      int stride)
      : offsets(off), order(ord), per_group(per_group_units), num(num_units), step(stride), first(first_unit),
        round(0), g(0), rem(0), r0(0), r1(0) {
    u = unit_of(0);
    if (u < num) {
      g = __ldg(order + u / per_group);
      rem = u % per_group;
      r0 = __ldg(offsets + g);
      r1 = __ldg(offsets + g + 1);
    }
    prefetch();
  }
  __device__ bool live() const { return u < num; }
  __device__ void prefetch() {
    un = unit_of(round + 1);
    gn = 0;
    r0n = r1n = 0;
    if (un < num) {
      gn = __ldg(order + un / per_group);
      r0n = __ldg(offsets + gn);
      r1n = __ldg(offsets + gn + 1);
    }
  }
  __device__ void next() {
    ++round;
    u = un;
    g = gn;
    rem = u % per_group;
    r0 = r0n;
    r1 = r1n;
    prefetch();
  }
};

template <int BN>
struct TgmmTile {
  static constexpr int kBoxBytes = kChunk * 64 * 2;  // 64 rows x 64 bf16 = 8 KB
  static constexpr int kABytes = 2 * kBoxBytes;      // 128 k columns
  static constexpr int kBBytes = (BN / 64) * kBoxBytes;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;
  // epilogue staging: one row of BN/2 bf16 per epilogue thread, padded by 16
  // bytes so a warp's 16-byte stores hit distinct banks
  // one 32-row x 64-column bf16 box (4 KB) per epilogue warp
  static constexpr int kStagingBytes = kEpiWarps * 4096;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + 256;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tgmm_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_dy,
                const __grid_constant__ CUtensorMap map_dw,
                const TgmmArgs args) {
  using C = TgmmTile<BN>;
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
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_dy);
    tma_prefetch_desc(&map_dw);
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

  const bool valid_meta = args.meta[kWsValid] != 0;
  const int KT = args.K / 128, NT = args.N / BN, KTNT = KT * NT;
  // G * KT * NT < 2^31 (checked by the host)
  const int num_units = valid_meta ? args.G * KTNT : 0;
  const int* offsets = args.meta + kWsOffsets;
  const uint64_t lim = args.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t c = 0;
      bool ok = true;
      UnitWalk w(offsets, args.order, KTNT, num_units, blockIdx.x, gridDim.x);
      for (; w.live() && ok; w.next()) {
        const int rem = w.rem;
        const int k0 = (rem / NT) * 128, n0 = (rem % NT) * BN;
        const int r0 = w.r0, r1 = w.r1;
        for (int r = r0; r < r1; r += kChunk) {
          const uint32_t s = c % kStages, ph = (c / kStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_word, lim)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = ring + s * C::kStageBytes;
          uint8_t* b_dst = a_dst + C::kABytes;
          mbar_arrive_expect_tx(&full[s], C::kStageBytes);
          tma_load_2d(a_dst, &map_x, &full[s], k0, r);
          tma_load_2d(a_dst + C::kBoxBytes, &map_x, &full[s], k0 + 64, r);
#pragma unroll
          for (int i = 0; i < BN / 64; ++i) tma_load_2d(b_dst + i * C::kBoxBytes, &map_dy, &full[s], n0 + 64 * i, r);
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
    // the whole warp walks the loop: lanes help zero foreign rows
    constexpr uint32_t idesc = make_idesc(1u /*bf16*/, true, true, kBM, BN);
    uint32_t c = 0, t = 0;
    bool ok = true;
    UnitWalk w(offsets, args.order, KTNT, num_units, blockIdx.x, gridDim.x);
    for (; w.live() && ok; w.next()) {
      const int r0 = w.r0, r1 = w.r1;
      if (r1 <= r0) continue;  // empty group: the epilogue writes zeros
      const uint32_t b = t & 1u, tph = (t >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty[b], tph ^ 1u, abort_word, lim))) break;
      tc_fence_after();
      const uint32_t d = tbase + b * BN;
      for (int r = r0; r < r1; r += kChunk) {
        const uint32_t s = c % kStages, ph = (c / kStages) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, abort_word, lim))) {
          ok = false;
          break;
        }
        uint8_t* a_ptr = ring + s * C::kStageBytes;
        uint8_t* b_ptr = a_ptr + C::kABytes;
        // rows of this chunk that belong to group g; the 16-row MMA steps past
        // them are skipped and the rest of the last step's rows (the next
        // group's) are zeroed in both x boxes (128 bytes per row and box)
        const int live = r1 - r;
        const int steps = live < kChunk ? (live + 15) / 16 : 4;
        if (live < 16 * steps) {
          const int words = (16 * steps - live) * 8;  // 16-byte words per box
          for (int i = 0; i < 2; ++i) {
            uint4* p = reinterpret_cast<uint4*>(a_ptr + i * C::kBoxBytes + live * 128);
            for (int w = lane; w < words; w += 32) p[w] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t a_addr = smem_u32(a_ptr);
          const uint32_t b_addr = smem_u32(b_ptr);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j < steps)
              mma_bf16(d, smem_desc_sw128(a_addr + 2048 * j, C::kBoxBytes, 1024),
                       smem_desc_sw128(b_addr + 2048 * j, C::kBoxBytes, 1024), idesc, (r > r0 || j > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        __syncwarp();
        ++c;
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&tfull[b]);
      __syncwarp();
      ++t;
    }
    if (lane == 0 && c > 0) {
      volatile int no_abort = 0;
      mma_commit(drain);
      mbar_wait(drain, 0, &no_abort, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    const int pw = warp - 2;
    const int h = pw >> 2;
    const int quad = warp & 3;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    uint8_t* box = staging + pw * 4096;
    uint8_t* brow = box + lane * 128;  // this thread's row of the box
    uint32_t t = 0;
    UnitWalk w(offsets, args.order, KTNT, num_units, blockIdx.x, gridDim.x);
    for (; w.live(); w.next()) {
      const int g = w.g;
      const int rem = w.rem;
      const int k0 = (rem / NT) * 128, n0 = (rem % NT) * BN;
      const int r0 = w.r0, r1 = w.r1;
      const int y = g * args.K + k0 + quad * 32;
      uint32_t r[BN / 2];
      if (r1 <= r0) {
#pragma unroll
        for (int j = 0; j < BN / 2; ++j) r[j] = 0u;
      } else {
        const uint32_t b = t & 1u, tph = (t >> 1) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[b], tph, abort_word, lim))) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < BN / 64; ++cc)
          tmem_ld_32x32(t_lane + b * BN + h * (BN / 2) + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * cc));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
        ++t;
      }
      // one 64-column box per pass; 16-byte chunk j of a row sits at chunk
      // position j ^ (row & 7) (the 128-byte swizzle of the dW tensor map)
#pragma unroll
      for (int pass = 0; pass < BN / 128; ++pass) {
        if (lane == 0) bulk_wait_read_all();  // the previous store has read the box
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = 64 * pass + 8 * j;
          *reinterpret_cast<uint4*>(brow + ((j ^ (lane & 7)) << 4)) =
              make_uint4(pack_bf16x2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])),
                         pack_bf16x2(__uint_as_float(r[c + 2]), __uint_as_float(r[c + 3])),
                         pack_bf16x2(__uint_as_float(r[c + 4]), __uint_as_float(r[c + 5])),
                         pack_bf16x2(__uint_as_float(r[c + 6]), __uint_as_float(r[c + 7])));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&map_dw, box, n0 + h * (BN / 2) + 64 * pass, y);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_word) atomicOr(const_cast<int32_t*>(args.meta) + kWsStatus, kErrTimeout);
}

// ---------------------------------------------------------------------------
// CTA-pair variant (K a multiple of 256).  A cluster of two CTAs on the two
// SMs of a pair owns the output tile (g, 256 rows of K, BN columns): each CTA
// loads its own 128 k columns of x and half (BN/2) of the dy columns of every
// 64-row chunk, and the even CTA issues one M=256 tcgen05.mma (cta_group::2)
// per 16-row step over both CTAs' shared memory; each CTA's TMEM receives its
// 128 k rows x BN.  A chunk takes 32 KB of each CTA's shared memory instead
// of 48 KB, so the ring holds six chunks instead of four.
//   warp 0     TMA producer (each CTA, its own halves into its own shared
//              memory).  The even CTA's full[s] takes two arrivals: its own
//              (with its bytes) and the odd CTA's, which for a whole chunk
//              registers its bytes remotely and lets its copies complete on
//              that barrier directly.
//   warp 1     even CTA: wait full[s], zero the next group's x rows of a
//              partial last step, issue the MMAs; commits arrive on both
//              CTAs' empty[s] / tfull[b].  Odd CTA: a chunk whose last step
//              holds rows of the next group lands on a local barrier; this
//              warp zeroes those rows and then arrives on the even CTA's
//              full[s].
//   warps 2-9  epilogue (each CTA, its 128 k rows); the odd CTA's warps free
//              the pair's TMEM buffer by remote arrives on the even CTA.
//   warp 10    even CTA: the pair's scheduler (below).
// Scheduling: the units are numbered largest groups first and the pairs
// claim them from a counter in the workspace as they go (list scheduling; a
// pair that runs slower, or drew larger units, takes fewer).  With skewed
// group sizes the claims alternate between the large and the small end of
// that order, so that long, read-heavy units and short, store-heavy ones run
// side by side.  The scheduler claims only while few chunks are queued ahead
// of its producer (several small units per claim once the units get small)
// and puts each unit {g, rem, r0, r1} in a queue of kQueue entries in its own
// shared memory and, by a bulk copy that completes on the odd CTA's barrier,
// in the odd CTA's.  Every role of both CTAs takes the units from
// its queue in the same order and frees an entry on the even CTA once it has
// read it.  The last CTA to finish resets the counters for the next launch.
constexpr int kPairStages = 6;  // default ring slots with BN = 256 (4 or 5 selectable)
constexpr int kPairThreads = 352;
constexpr int kSchedWarp = 10;
constexpr int kQueue = 16;
constexpr int kQueueReaders = 2 * (2 + kEpiWarps);  // producer, warp 1, epilogue warps; both CTAs
// the scheduler holds at most TgmmArgs::claim_ahead units (default 3) beyond
// those the even CTA's producer has taken, claims only while fewer than 8
// chunks are queued ahead of that producer, and takes up to
// TgmmArgs::max_batch (1..kMaxBatch, default 4) small units per claim

// Zero rows [from, to) of both 64-row x boxes of a ring slot (128 bytes per
// row and box, so the swizzle does not matter) and fence them into the async
// proxy; the warp's lanes share the stores.
__device__ __forceinline__ void zero_x_rows(uint8_t* a_ptr, int from, int to, int lane) {
  constexpr int kBox = kChunk * 64 * 2;
  const int words = (to - from) * 8;
  for (int i = 0; i < 2; ++i) {
    uint4* p = reinterpret_cast<uint4*>(a_ptr + i * kBox + from * 128);
    for (int q = lane; q < words; q += 32) p[q] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
}

template <int BN, int STAGES>
struct TgmmPairTile {
  static constexpr int kBoxBytes = kChunk * 64 * 2;           // 64 rows x 64 bf16 = 8 KB
  static constexpr int kABytes = 2 * kBoxBytes;               // this CTA's 128 k columns
  static constexpr int kBBytes = (BN / 2 / 64) * kBoxBytes;   // this CTA's BN/2 n columns
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = STAGES;  // kPairStages (or 4, 5) with BN = 256; 8 with BN = 128
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kStagingBytes = kEpiWarps * 4096;
  // queue entries (16 bytes each), then the barriers, the TMEM address and the abort word
  static constexpr int kTailBytes = 16 * kQueue + 8 * (3 * kStages + 5 + 2 * kQueue) + 16;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + 1024;
  static_assert(kTailBytes <= 1024, "barrier area");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Entry i of a CTA's unit queue (every lane of the calling warp, or the one
// thread of a single-thread role, with `warp_wide` false); the entry is freed
// on the even CTA as soon as it has been read.
struct UnitQueue {
  uint64_t* full;
  uint64_t* empty;
  const int4* data;
  uint32_t empty_leader;  // shared::cluster address of the even CTA's empty[0]
  bool leader;
  __device__ bool get(uint32_t i, int4& e, bool warp_wide, int lane, volatile int* abort_word,
                      uint64_t lim) const {
    const uint32_t slot = i % kQueue, ph = (i / kQueue) & 1u;
    bool ok = mbar_wait(&full[slot], ph, abort_word, lim);
    if (warp_wide) ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    e = data[slot];
    if (warp_wide) __syncwarp();
    if (lane == 0) {
      if (leader)
        mbar_arrive(&empty[slot]);
      else
        mbar_arrive_remote(empty_leader + slot * 8u);
    }
    return true;
  }
};

template <int BN, int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    tgmm_pair_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_dy,
                     const __grid_constant__ CUtensorMap map_dw, const TgmmArgs args) {
  using C = TgmmPairTile<BN, STAGES>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  uint8_t* staging = smem + S * C::kStageBytes;
  int4* qdata = reinterpret_cast<int4*>(staging + C::kStagingBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(qdata + kQueue);  // even CTA: both halves ready
  uint64_t* ploaded = full + S;  // odd CTA: a chunk to be zeroed landed
  uint64_t* empty = ploaded + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;      // even CTA: both CTAs' epilogues freed buffer b
  uint64_t* drain = tempty + 2;
  uint64_t* qfull = drain + 1;       // each CTA: queue entry written
  uint64_t* qempty = qfull + kQueue;  // even CTA: every reader of both CTAs has read the entry
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qempty + kQueue);
  volatile int* abort_word = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* taken = abort_word + 1;  // even CTA: queue entries its producer has taken
  volatile int* ctaken = taken + 1;      // even CTA: chunks its producer has issued (1 per empty unit)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    *taken = 0;
    *ctaken = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);
      mbar_init(&ploaded[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    for (int q = 0; q < kQueue; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], kQueueReaders);
    }
    *abort_word = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_dy);
    tma_prefetch_desc(&map_dw);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();  // inputs, metadata and the work counter come from earlier kernels

  const bool valid_meta = args.meta[kWsValid] != 0;
  const int KP = args.K / 256, NT = args.N / BN, KPNT = KP * NT;
  const int num_units = valid_meta ? args.G * KPNT : 0;
  const int* offsets = args.meta + kWsOffsets;
  const uint64_t lim = args.wait_limit_ns;
  const UnitQueue queue{qfull, qempty, qdata, mapa_shared(smem_u32(qempty), 0), leader};

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);
      uint32_t c = 0;
      bool ok = true;
      int4 e;
      int issued = 0;
      for (uint32_t i = 0; ok && queue.get(i, e, false, 0, abort_word, lim) && e.x >= 0; ++i) {
        *taken = static_cast<int>(i) + 1;
        const int rem = e.y, r0 = e.z, r1 = e.w;
        if (r1 <= r0) *ctaken = ++issued;  // an empty group's unit counts as one chunk
        const int k0 = (rem / NT) * 256 + static_cast<int>(rank) * 128;
        const int n0 = (rem % NT) * BN + static_cast<int>(rank) * (BN / 2);
        for (int r = r0; r < r1; r += kChunk) {
          const uint32_t s = c % S, ph = (c / S) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_word, lim)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = ring + s * C::kStageBytes;
          uint8_t* b_dst = a_dst + C::kABytes;
          const int live = r1 - r;
          const bool zero = live < kChunk && (live & 15) != 0;  // last step holds next-group rows
          if (leader || zero) {
            // local completion: the even CTA's own half, or an odd-CTA chunk
            // that warp 1 must zero before it counts
            uint64_t* bar = leader ? &full[s] : &ploaded[s];
            mbar_arrive_expect_tx(bar, C::kStageBytes);
            tma_load_2d(a_dst, &map_x, bar, k0, r);
            tma_load_2d(a_dst + C::kBoxBytes, &map_x, bar, k0 + 64, r);
#pragma unroll
            for (int i2 = 0; i2 < BN / 128; ++i2)
              tma_load_2d(b_dst + i2 * C::kBoxBytes, &map_dy, bar, n0 + 64 * i2, r);
          } else {
            // completes on the even CTA's barrier; the bytes may land before
            // the expectation is registered (the count dips below zero
            // within the phase)
            const uint32_t bar = full0 + s * 8u;
            mbar_arrive_expect_tx_remote(bar, C::kStageBytes);
            tma_load_2d_pair(a_dst, &map_x, bar, k0, r);
            tma_load_2d_pair(a_dst + C::kBoxBytes, &map_x, bar, k0 + 64, r);
#pragma unroll
            for (int i2 = 0; i2 < BN / 128; ++i2)
              tma_load_2d_pair(b_dst + i2 * C::kBoxBytes, &map_dy, bar, n0 + 64 * i2, r);
          }
          ++c;
          *ctaken = ++issued;
        }
      }
      // the even CTA waits for the last copies into every slot (they land in
      // microseconds); the odd CTA's copies land before the even CTA's MMAs
      // read them, so before the pair passes the teardown cluster barrier
      volatile int no_abort = 0;
      for (uint32_t s = 0; leader && s < S; ++s) {
        if (c > s) {
          const uint32_t last = s + S * ((c - 1 - s) / S);
          mbar_wait(&full[s], (last / S) & 1u, &no_abort, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1 && leader) {
    constexpr uint32_t idesc = make_idesc(1u /*bf16*/, true, true, 2 * kBM, BN);
    uint32_t c = 0, t = 0;
    bool ok = true;
    int4 e;
    for (uint32_t i = 0; ok && queue.get(i, e, true, lane, abort_word, lim) && e.x >= 0; ++i) {
      const int r0 = e.z, r1 = e.w;
      if (r1 <= r0) continue;  // empty group: the epilogues write zeros
      const uint32_t b = t & 1u, tph = (t >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty[b], tph ^ 1u, abort_word, lim))) break;
      tc_fence_after();
      const uint32_t d = tbase + b * BN;
      for (int r = r0; r < r1; r += kChunk) {
        const uint32_t s = c % S, ph = (c / S) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, abort_word, lim))) {
          ok = false;
          break;
        }
        uint8_t* a_ptr = ring + s * C::kStageBytes;
        uint8_t* b_ptr = a_ptr + C::kABytes;
        const int live = r1 - r;
        const int steps = live < kChunk ? (live + 15) / 16 : 4;
        if (live < 16 * steps) zero_x_rows(a_ptr, live, 16 * steps, lane);
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t a_addr = smem_u32(a_ptr);
          const uint32_t b_addr = smem_u32(b_ptr);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j < steps)
              mma_bf16_pair(d, smem_desc_sw128(a_addr + 2048 * j, C::kBoxBytes, 1024),
                            smem_desc_sw128(b_addr + 2048 * j, C::kBoxBytes, 1024), idesc,
                            (r > r0 || j > 0) ? 1u : 0u);
          }
          mma_commit_pair(&empty[s], 0x3);
        }
        __syncwarp();
        ++c;
      }
      if (!ok) break;
      if (lane == 0) mma_commit_pair(&tfull[b], 0x3);
      __syncwarp();
      ++t;
    }
    if (lane == 0 && c > 0) {
      volatile int no_abort = 0;
      mma_commit_pair(drain, 0x1);
      mbar_wait(drain, 0, &no_abort, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // odd CTA: zero the next group's x rows of partial chunks, then count
    // them on the even CTA's full[s]
    const uint32_t full0 = mapa_shared(smem_u32(full), 0);
    uint32_t c = 0, pp = 0;  // pp: parity of ploaded[s], one bit per slot
    bool ok = true;
    int4 e;
    for (uint32_t i = 0; ok && queue.get(i, e, true, lane, abort_word, lim) && e.x >= 0; ++i) {
      for (int r = e.z; r < e.w; r += kChunk, ++c) {
        const int live = e.w - r;
        if (!(live < kChunk && (live & 15) != 0)) continue;
        const uint32_t s = c % S;
        if (!__all_sync(0xffffffffu, mbar_wait(&ploaded[s], (pp >> s) & 1u, abort_word, lim))) {
          ok = false;
          break;
        }
        pp ^= 1u << s;
        zero_x_rows(ring + s * C::kStageBytes, live, (live + 15) & ~15, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(full0 + s * 8u);
      }
    }
  } else if (warp < kSchedWarp) {
    const int pw = warp - 2;
    const int h = pw >> 2;
    const int quad = warp & 3;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
    uint8_t* box = staging + pw * 4096;
    uint8_t* brow = box + lane * 128;
    uint32_t t = 0;
    int4 e;
    for (uint32_t i = 0; queue.get(i, e, true, lane, abort_word, lim) && e.x >= 0; ++i) {
      const int g = e.x;
      const int rem = e.y;
      const int k0 = (rem / NT) * 256 + static_cast<int>(rank) * 128, n0 = (rem % NT) * BN;
      const int r0 = e.z, r1 = e.w;
      const int y = g * args.K + k0 + quad * 32;
      uint32_t r[BN / 2];
      if (r1 <= r0) {
#pragma unroll
        for (int j = 0; j < BN / 2; ++j) r[j] = 0u;
      } else {
        const uint32_t b = t & 1u, tph = (t >> 1) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[b], tph, abort_word, lim))) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < BN / 64; ++cc)
          tmem_ld_32x32(t_lane + b * BN + h * (BN / 2) + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * cc));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty0 + b * 8u);
        ++t;
      }
#pragma unroll
      for (int pass = 0; pass < BN / 128; ++pass) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int cidx = 64 * pass + 8 * j;
          *reinterpret_cast<uint4*>(brow + ((j ^ (lane & 7)) << 4)) =
              make_uint4(pack_bf16x2(__uint_as_float(r[cidx]), __uint_as_float(r[cidx + 1])),
                         pack_bf16x2(__uint_as_float(r[cidx + 2]), __uint_as_float(r[cidx + 3])),
                         pack_bf16x2(__uint_as_float(r[cidx + 4]), __uint_as_float(r[cidx + 5])),
                         pack_bf16x2(__uint_as_float(r[cidx + 6]), __uint_as_float(r[cidx + 7])));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&map_dw, box, n0 + h * (BN / 2) + 64 * pass, y);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
  } else if (leader && lane == 0) {
    // ------------------------------------------------------------ scheduler
    int* claimed = const_cast<int32_t*>(args.meta) + kWsClaimed;
    const uint32_t odd_full = mapa_shared(smem_u32(qfull), 1);
    const uint32_t odd_data = mapa_shared(smem_u32(qdata), 1);
    uint32_t i = 0;
    auto publish = [&](int4 v) -> bool {
      const uint32_t slot = i % kQueue, ph = (i / kQueue) & 1u;
      // no more than claim_ahead entries beyond the producer (bounded wait)
      if (*taken + args.claim_ahead <= static_cast<int>(i)) {
        const uint64_t t0 = global_timer_ns();
        while (*taken + args.claim_ahead <= static_cast<int>(i)) {
          if (*abort_word) return false;
          if (global_timer_ns() - t0 > lim) {
            *abort_word = 1;
            return false;
          }
          __nanosleep(64);
        }
      }
      if (!mbar_wait(&qempty[slot], ph ^ 1u, abort_word, lim)) return false;
      qdata[slot] = v;
      fence_proxy_async_smem();  // the bulk copy reads the entry through the async proxy
      mbar_arrive_expect_tx_remote(odd_full + slot * 8u, 16);
      bulk_copy_s2cluster(odd_data + slot * 16u, &qdata[slot], 16, odd_full + slot * 8u);
      mbar_arrive(&qfull[slot]);
      ++i;
      return true;
    };
    constexpr int kMaxBatch = 4;
    // Claim q takes unit q/2 from the large end of the size order when q is
    // even and unit num_units-1-q/2 from the small end when q is odd, so every
    // pair alternates long, read-heavy units with short ones whose cost is
    // mostly the dW store (or only that, for an empty group): the loads of the
    // one overlap the stores of the other, and the launch never runs a phase of
    // loads only followed by a phase of stores only.
    // With groups of about one size there is nothing to mix, and the plain
    // order keeps each group's units together: alternate only when the
    // largest group has more than twice the chunks of the smallest.
    bool mix = false;
    if (num_units > 0) {
      const int gl = __ldg(args.order), gs = __ldg(args.order + args.G - 1);
      const int cl = (__ldg(offsets + gl + 1) - __ldg(offsets + gl) + kChunk - 1) / kChunk;
      const int cs = (__ldg(offsets + gs + 1) - __ldg(offsets + gs) + kChunk - 1) / kChunk;
      mix = cl > 2 * cs;
    }
    auto unit_of = [&](int q) { return (mix && (q & 1)) ? num_units - 1 - (q >> 1) : (mix ? (q >> 1) : q); };
    // Claims are paced by work: the next claim is made only once the producer
    // is within kLeadChunks chunks of the end of what is already published, so
    // that a claimed unit starts within a few microseconds (the units of one
    // group, claimed one after the other, then read its rows at about the same
    // time and find them in L2, instead of one of them waiting behind a long
    // unit and reading them again after they were evicted).
    constexpr int kLeadChunks = 8;
    bool ok = true;
    int batch = min(mix ? 2 : 1, args.max_batch);
    int published = 0;  // chunks of the published units (1 for an empty group's)
    while (ok) {
      if (published - *ctaken >= kLeadChunks) {
        const uint64_t t0 = global_timer_ns();
        while (published - *ctaken >= kLeadChunks) {
          if (*abort_word || global_timer_ns() - t0 > lim) break;
          __nanosleep(64);
        }
        if (*abort_word || published - *ctaken >= kLeadChunks) {
          *abort_word = 1;
          ok = false;
          break;
        }
      }
      const int k0 = atomicAdd(claimed, batch);
      if (k0 >= num_units) break;
      const int cnt = min(batch, num_units - k0);
      int u[kMaxBatch], g[kMaxBatch], r0[kMaxBatch], r1[kMaxBatch];
#pragma unroll
      for (int j = 0; j < kMaxBatch; ++j) u[j] = j < cnt ? unit_of(k0 + j) : 0;
#pragma unroll
      for (int j = 0; j < kMaxBatch; ++j) g[j] = j < cnt ? __ldg(args.order + u[j] / KPNT) : 0;
#pragma unroll
      for (int j = 0; j < kMaxBatch; ++j) {
        r0[j] = j < cnt ? __ldg(offsets + g[j]) : 0;
        r1[j] = j < cnt ? __ldg(offsets + g[j] + 1) : 0;
      }
#pragma unroll
      for (int j = 0; j < kMaxBatch; ++j) {
        if (ok && j < cnt) {
          ok = publish(make_int4(g[j], u[j] % KPNT, r0[j], r1[j]));
          published += max(1, (r1[j] - r0[j] + kChunk - 1) / kChunk);
        }
      }
      // the large-end units shrink as the claims go on: claim more at once
      // when they get small (when mixing, the first claim of the batch is a
      // large-end one whenever the batch size is even)
      const int jf = (mix && (k0 & 1)) ? (cnt > 1 ? 1 : 0) : 0;
      const int chunks = (r1[jf] - r0[jf] + kChunk - 1) / kChunk;
      batch = min(chunks >= 4 ? (mix ? 2 : 1) : chunks >= 2 ? 2 : 4, args.max_batch);
    }
    if (ok) publish(make_int4(-1, 0, 0, 0));
  }

  // teardown: no CTA of the pair leaves while the other may still arrive on
  // its barriers or its MMAs may still touch the other's TMEM
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, C::kTmemCols);
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

template <int BN, int STAGES>
cudaError_t launch_pair(const CUtensorMap& map_x, const CUtensorMap& map_dy, const CUtensorMap& map_dw,
                        const TgmmArgs& args, int max_pairs, cudaStream_t stream) {
  constexpr int smem = TgmmPairTile<BN, STAGES>::kSmemBytes;
  auto kernel = tgmm_pair_kernel<BN, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // as many pairs as can be resident at once (one CTA per SM)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * max_pairs, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int pairs = clusters < max_pairs ? clusters : max_pairs;
  return launch_pdl(kernel, dim3(2 * pairs), dim3(kPairThreads), smem, stream, map_x, map_dy, map_dw, args);
}

template <int BN>
cudaError_t launch(const CUtensorMap& map_x, const CUtensorMap& map_dy, const CUtensorMap& map_dw,
                   const TgmmArgs& args, int grid,
                   cudaStream_t stream) {
  constexpr int smem = TgmmTile<BN>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(tgmm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(tgmm_kernel<BN>, dim3(grid), dim3(kThreads), smem, stream, map_x, map_dy, map_dw, args);
}

}  // namespace

int tgmm_bn(int N) { return (N % 256 == 0) ? 256 : 128; }

cudaError_t launch_tgmm_bf16(const CUtensorMap& map_x, const CUtensorMap& map_dy, const CUtensorMap& map_dw,
                             const TgmmArgs& args, int grid,
                             cudaStream_t stream) {
  if (args.K % 256 == 0) {
    // CTA pairs: grid / 2 pairs at most (grid = min(SMs, tiles))
    const int max_pairs = grid / 2 > 0 ? grid / 2 : 1;
    if (args.N % 256 == 0) {
      if (args.stages == 4) return launch_pair<256, 4>(map_x, map_dy, map_dw, args, max_pairs, stream);
      if (args.stages == 5) return launch_pair<256, 5>(map_x, map_dy, map_dw, args, max_pairs, stream);
      return launch_pair<256, kPairStages>(map_x, map_dy, map_dw, args, max_pairs, stream);
    }
    return launch_pair<128, 8>(map_x, map_dy, map_dw, args, max_pairs, stream);
  }
  if (args.N % 256 == 0) return launch<256>(map_x, map_dy, map_dw, args, grid, stream);
  return launch<128>(map_x, map_dy, map_dw, args, grid, stream);
}

}  // namespace gmm
