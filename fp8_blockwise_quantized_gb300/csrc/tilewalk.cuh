// The CTA-pair FP8 kernel's static walk over its work units (the single-CTA
// kernel claims its units from a counter instead).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace gmm {

// A CTA (or CTA pair) takes units u = first, first + step, ...: tile u / per_tile
// and column block u % per_tile (row-tile major), or tile u % num_tiles and
// column block u / num_tiles (column-block major).  The next unit's tile is
// loaded one unit ahead, so its global-memory latency overlaps the current
// unit instead of sitting between two units on each role's path.  The host
// keeps the number of units below 2^31, so unit indices are 32-bit.
struct TileWalk {
  const Tile* tiles;
  uint32_t num, u, d, step;  // d: per_tile (row-tile major) or num_tiles (column-block major)
  bool col_major;
  Tile cur, nxt;
  __device__ TileWalk(const Tile* t, uint32_t per_tile, uint32_t num_units, uint32_t num_tiles, bool column_major,
                      uint32_t first, uint32_t stride)
      : tiles(t), num(num_units), u(first), d(column_major ? num_tiles : per_tile), step(stride),
        col_major(column_major) {
    if (u < num) cur = load(u);
    prefetch();
  }
  __device__ Tile load(uint32_t v) const {
    const int4 q = __ldg(reinterpret_cast<const int4*>(tiles + (col_major ? v % d : v / d)));
    return Tile{q.x, q.y, q.z, q.w};
  }
  __device__ void prefetch() {
    const uint32_t un = u + step;
    if (un < num) nxt = load(un);
  }
  __device__ bool live() const { return u < num; }
  __device__ int col0(int cols) const { return static_cast<int>(col_major ? u / d : u % d) * cols; }
  __device__ void next() {
    u += step;
    cur = nxt;
    prefetch();
  }
};

}  // namespace gmm
