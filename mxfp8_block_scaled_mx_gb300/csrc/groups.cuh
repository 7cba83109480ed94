// groups.cuh -- device-side group bookkeeping shared by the grouped
// quantizer and the grouped GEMM.  Group offsets live in device memory and
// are read by every block, so no host synchronization is needed.
#pragma once

#include <cstdint>

namespace mx {

constexpr int kMaxGroups = 1000;

// Warp 0 of the block copies offsets o[0..groups] into s_off and writes
// s_tiles[g] = sum_{h<g} ceil((o[h+1] - o[h]) / 128) for g = 0..groups, the
// number of 128-row tiles (= padded scale row tiles) before group g, and,
// when s_units is not null, s_units[g] = sum_{h<g} ceil(tiles_h / cm), the
// number of cm-tile units (tiles of one block cluster) before group g.  It
// validates 0 = o[0] <= o[1] <= ... <= o[groups] = total and stores the
// verdict in *s_valid.  The caller synchronizes the block afterwards.
__device__ __forceinline__ void group_tile_prefix(const int32_t* __restrict__ offsets, int groups,
                                                  int64_t total, int32_t* s_off, int32_t* s_tiles,
                                                  int32_t* s_valid, int cm = 1,
                                                  int32_t* s_units = nullptr) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int32_t carry = 0, carry_u = 0;
  bool ok = true;
  for (int base = 0; base < groups; base += 32) {
    const int g = base + lane;
    int32_t tiles = 0;
    if (g < groups) {
      const int32_t lo = offsets[g];
      const int32_t hi = offsets[g + 1];
      s_off[g] = lo;
      if (hi < lo) ok = false;
      tiles = hi > lo ? (hi - lo + 127) / 128 : 0;
    }
    int32_t incl = tiles;
    int32_t incl_u = (tiles + cm - 1) / cm;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
      const int32_t vu = __shfl_up_sync(0xffffffffu, incl_u, d);
      if (lane >= d) {
        incl += v;
        incl_u += vu;
      }
    }
    if (g < groups) {
      s_tiles[g + 1] = carry + incl;
      if (s_units) s_units[g + 1] = carry_u + incl_u;
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
    carry_u += __shfl_sync(0xffffffffu, incl_u, 31);
  }
  if (lane == 0) {
    const int32_t first = offsets[0];
    const int32_t last = offsets[groups];
    s_off[groups] = last;
    s_tiles[0] = 0;
    if (s_units) s_units[0] = 0;
    if (first != 0 || static_cast<int64_t>(last) != total) ok = false;
  }
  ok = __all_sync(0xffffffffu, ok);
  if (lane == 0) *s_valid = ok ? 1 : 0;
}

// Largest g in [0, groups) with s_tiles[g] <= t (t < s_tiles[groups]).
// Because empty groups repeat a prefix value, the largest such g is the
// non-empty group that owns tile t.
__device__ __forceinline__ int find_group(const int32_t* s_tiles, int groups, int32_t t) {
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tiles[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

}  // namespace mx
