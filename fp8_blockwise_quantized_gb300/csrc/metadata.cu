// a1: group metadata on the device.
//
// Rows are sorted by expert into contiguous groups ("MoE 优化的探索", §3.7.2);
// a grouped kernel finds each tile's expert through offsets and a tile list
// built from group_sizes on the device ("实现差距：GMM Kernel（V1 vs V2）", §1
// and §2.2: the metadata is filled inside the kernel, not on the host).
//
// One CTA of 1024 threads: each thread owns a contiguous run of at most
// ceil(G/1024) groups, the block scans the per-thread row and tile counts, and
// every thread then writes its groups' offsets, 128-row tiles and 256-row
// tiles (the row tiles of the CTA-pair FP8 kernel).
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace gmm {

namespace {

template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    T o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

// Exclusive scan over the block (1024 threads); returns the block total in *total.
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* warp_sums,
                                                          long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long inc = warp_inclusive_scan(v);
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    long long w = warp_sums[lane];
    long long winc = warp_inclusive_scan(w);
    warp_sums[lane] = winc - w;  // exclusive prefix of the warp totals
    if (lane == 31) warp_sums[32] = winc;
  }
  __syncthreads();
  long long r = inc - v + warp_sums[warp];
  *total = warp_sums[32];
  __syncthreads();
  return r;
}

}  // namespace

__global__ void __launch_bounds__(1024) group_metadata_kernel(const int32_t* __restrict__ sizes, int G,
                                                                int M, int32_t* __restrict__ ws,
                                                                Tile* __restrict__ tiles,
                                                                int32_t* __restrict__ order,
                                                                Tile* __restrict__ pair_tiles) {
  __shared__ long long warp_sums[33];
  __shared__ unsigned long long keys[kMaxGroups];
  griddep_launch_dependents();
  griddep_wait();  // group_sizes may come from the previous kernel
  const int t = threadIdx.x;
  const int per = (G + 1023) / 1024;
  const int g0 = min(G, t * per), g1 = min(G, g0 + per);

  long long rows = 0, ntiles = 0, npairs = 0;
  int bad = 0;
  for (int g = g0; g < g1; ++g) {
    const int n = sizes[g];
    if (n < 0) {
      bad = 1;
    } else {
      rows += n;
      ntiles += (n + kBM - 1) / kBM;
      npairs += (n + 2 * kBM - 1) / (2 * kBM);
    }
  }
  const int any_bad = __syncthreads_or(bad);
  long long rows_total, tiles_total, pairs_total;
  const long long row_off = block_exclusive_scan(rows, warp_sums, &rows_total);
  const long long tile_off = block_exclusive_scan(ntiles, warp_sums, &tiles_total);
  const long long pair_off = block_exclusive_scan(npairs, warp_sums, &pairs_total);

  int err = 0;
  if (any_bad) err |= kErrNegativeGroup;
  else if (rows_total > M) err |= kErrGroupsExceedM;

  if (err == 0) {
    long long off = row_off, tix = tile_off, pix = pair_off;
    for (int g = g0; g < g1; ++g) {
      const int n = sizes[g];
      ws[kWsOffsets + g] = static_cast<int>(off);
      for (int r = 0; r < n; r += kBM) {
        Tile tl;
        tl.g = g;
        tl.row0 = static_cast<int>(off + r);
        tl.row1 = static_cast<int>(off + min(n, r + kBM));
        tl.pad = 0;
        tiles[tix++] = tl;
      }
      for (int r = 0; r < n; r += 2 * kBM) {
        Tile tl;
        tl.g = g;
        tl.row0 = static_cast<int>(off + r);
        tl.row1 = static_cast<int>(off + min(n, r + 2 * kBM));
        tl.pad = 0;
        pair_tiles[pix++] = tl;
      }
      off += n;
    }
  }
  if (err == 0) {
    // the groups by size, descending, ties by index: group g's place is the
    // number of keys (INT32_MAX - size, index) below its own (all keys are
    // distinct), so each thread ranks its groups against all G keys, read as
    // shared-memory broadcasts.  The tgmm kernels deal the units of the
    // largest groups first, so that the last units of the grid are small.
    for (int i = t; i < G; i += blockDim.x)
      keys[i] = (static_cast<unsigned long long>(0x7fffffff - sizes[i]) << 32) | static_cast<unsigned>(i);
    __syncthreads();
    for (int i = t; i < G; i += blockDim.x) {
      const unsigned long long mine = keys[i];
      int rank = 0;
      for (int j = 0; j < G; ++j) rank += keys[j] < mine ? 1 : 0;
      order[rank] = i;
    }
  }
  if (t == 0) {
    ws[kWsClaimed] = 0;
    ws[kWsFinished] = 0;
    if (err) {
      atomicOr(ws + kWsStatus, err);
      ws[kWsValid] = 0;
      ws[kWsS] = M;
      ws[kWsNumTiles] = 0;
      ws[kWsNumPairTiles] = 0;
    } else {
      ws[kWsValid] = 1;
      ws[kWsS] = static_cast<int>(rows_total);
      ws[kWsNumTiles] = static_cast<int>(tiles_total);
      ws[kWsNumPairTiles] = static_cast<int>(pairs_total);
      ws[kWsOffsets + G] = static_cast<int>(rows_total);
    }
  }
}

cudaError_t launch_group_metadata(const int32_t* sizes, int G, int M, void* workspace, cudaStream_t stream) {
  char* base = static_cast<char*>(workspace);
  return launch_pdl(group_metadata_kernel, dim3(1), dim3(1024), 0, stream, sizes, G, M, static_cast<int32_t*>(workspace),
                    reinterpret_cast<Tile*>(base + tiles_offset_bytes(G)),
                    reinterpret_cast<int32_t*>(base + order_offset_bytes(G, M)),
                    reinterpret_cast<Tile*>(base + pair_tiles_offset_bytes(G, M)));
}

}  // namespace gmm
