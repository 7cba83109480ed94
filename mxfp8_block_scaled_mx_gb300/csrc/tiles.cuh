// tiles.cuh -- work decomposition of the block-pair GEMM kernel: the
// shared-memory group table, and the mapping of a linear work unit to one
// block's output tile, operand coordinates and scale units in the three
// GEMM modes (dense; grouped by rows of A; grouped along K).
#pragma once

#include <cstdint>

#include "groups.cuh"
#include "kernels.h"

namespace mx {

constexpr int kTileM = 128;   // output rows per block
constexpr int kTileK = 128;   // K elements (bytes) per pipeline stage = 4 scale blocks

struct GroupSmem {
  int32_t off[kMaxGroups + 1];
  int32_t tiles[kMaxGroups + 1];   // 128-row tiles before each group
  int32_t units[kMaxGroups + 1];   // cluster units (CM tiles) before each group
  int32_t valid;
};

struct TileInfo {
  int64_t m0;        // first row of the A tile
  int64_t y_row0;    // output row of the tile's first row
  int64_t m_end;     // output rows >= m_end are not stored
  int64_t n0;        // first column of Y (first row of the group's B)
  int64_t b_row0;    // first row of the B tile in the B tensor map
  int64_t a_kx0;     // first K column of the A operand in its tensor map
  int64_t b_kx0;     // first K column of the B operand
  int64_t sfa_unit;  // first 512-byte scale unit of A (-1: this block's tile is padding)
  int64_t sfb_unit;  // first scale unit of the B tile's first 128-row tile
  int64_t sfb_step;  // scale units between consecutive 128-row tiles of B
  int32_t k_blocks;  // 32-element K blocks of the tile's contraction (a partial
                     // final block, zero-filled past K by the tensor copy, counts)
  // The same scale units as (row tile, first K tile) coordinates of the
  // [row tiles][K tiles] unit grid (3-D tensor-map copies); sfa_rt is set
  // even for a padding tile (its scales are loaded and never used).
  int32_t sfa_rt, sfa_kt0, sfb_rt, sfb_kt0;
};

// Work unit u of a cluster = CM m-tiles x one n-tile; block `rank` of the
// cluster takes m-tile CM*mu + rank.  Dense units follow a banded raster
// (p.band_m m-tiles per band, n outer inside a band) so a band of A stays in
// L2 while B streams once per band; units grouped by rows walk groups, then
// m-units, then n; units grouped along K walk groups, then m-units, then n,
// every group covering the whole [m, n] output of its own matrix.  Scale
// units: 512 bytes per 128 rows x 128 K, ceil(ld / 128) per 128-row tile.
// The host keeps the unit count below 2^31, so the unit index arithmetic
// runs in 32 bits (a 64-bit division by a run-time value costs several
// hundred cycles on the epilogue's path between two tiles).
template <int BN, int MODE, int CM>
__device__ __forceinline__ TileInfo tile_info(const GemmParams& p, int64_t u, int64_t n_tiles,
                                              uint32_t rank, const GroupSmem* gs) {
  TileInfo ti;
  const int64_t a_tiles_k = (p.lda + 127) / 128;
  const int64_t b_tiles_k = (p.ldb + 127) / 128;
  ti.a_kx0 = 0;
  ti.b_kx0 = 0;
  ti.sfb_step = b_tiles_k;
  ti.k_blocks = static_cast<int32_t>((p.k + 31) / 32);
  const uint32_t u32 = static_cast<uint32_t>(u);
  const uint32_t nt32 = static_cast<uint32_t>(n_tiles);
  if constexpr (MODE == kModeGroupM) {
    const uint32_t mu32 = u32 / nt32;
    const int64_t mu = mu32;
    const int64_t n_blk = u32 - mu32 * nt32;
    const int g = find_group(gs->units, p.groups, static_cast<int32_t>(mu));
    const int64_t lm = (mu - gs->units[g]) * CM + rank;  // m-tile inside the group
    const int64_t g_tiles = gs->tiles[g + 1] - gs->tiles[g];
    ti.m0 = static_cast<int64_t>(gs->off[g]) + lm * kTileM;
    ti.y_row0 = ti.m0;
    ti.m_end = lm < g_tiles ? static_cast<int64_t>(gs->off[g + 1]) : ti.m0;
    ti.sfa_unit = lm < g_tiles ? (gs->tiles[g] + lm) * a_tiles_k : -1;
    ti.sfa_rt = static_cast<int32_t>(gs->tiles[g] + lm);
    ti.sfa_kt0 = 0;
    ti.n0 = n_blk * BN;
    if (p.b_concat) {
      // one [n, ldb] B; expert g's operand is columns [g*k, (g+1)*k)
      ti.b_row0 = ti.n0;
      ti.b_kx0 = static_cast<int64_t>(g) * p.k;
      ti.sfb_rt = static_cast<int32_t>(ti.n0 / 128);
      ti.sfb_kt0 = static_cast<int32_t>(static_cast<int64_t>(g) * (p.k / 128));
    } else {
      // [groups, n, k] B, one swizzled scale matrix per expert
      ti.b_row0 = static_cast<int64_t>(g) * p.n + ti.n0;
      ti.sfb_rt = static_cast<int32_t>(ti.b_row0 / 128);
      ti.sfb_kt0 = 0;
    }
    ti.sfb_unit = ti.sfb_rt * b_tiles_k + ti.sfb_kt0;
  } else if constexpr (MODE == kModeGroupK) {
    const int64_t m_tiles = (p.m + kTileM - 1) / kTileM;
    const uint32_t per_group = static_cast<uint32_t>((m_tiles + CM - 1) / CM) * nt32;
    const int g = static_cast<int>(u32 / per_group);
    const uint32_t w = u32 - static_cast<uint32_t>(g) * per_group;
    const uint32_t mu32 = w / nt32;
    const int64_t mu = mu32;
    const int64_t n_blk = w - mu32 * nt32;
    const int64_t m_blk = mu * CM + rank;
    const int64_t kt0 = gs->tiles[g];  // the group's first 128-column K tile
    ti.m0 = m_blk * kTileM;
    ti.y_row0 = static_cast<int64_t>(g) * p.m + ti.m0;
    ti.m_end = static_cast<int64_t>(g) * p.m + p.m;  // a padding m-tile starts past it
    ti.sfa_unit = m_blk < m_tiles ? m_blk * a_tiles_k + kt0 : -1;
    ti.sfa_rt = static_cast<int32_t>(m_blk);
    ti.sfa_kt0 = static_cast<int32_t>(kt0);
    ti.n0 = n_blk * BN;
    ti.b_row0 = ti.n0;
    ti.a_kx0 = kt0 * kTileK;
    ti.b_kx0 = kt0 * kTileK;
    ti.sfb_rt = static_cast<int32_t>(ti.n0 / 128);
    ti.sfb_kt0 = static_cast<int32_t>(kt0);
    ti.sfb_unit = ti.sfb_rt * b_tiles_k + kt0;
    ti.k_blocks = (gs->off[g + 1] - gs->off[g] + 31) / 32;
  } else {
    const int64_t m_tiles = (p.m + kTileM - 1) / kTileM;
    const int64_t m_units = (m_tiles + CM - 1) / CM;
    const uint32_t band_units = static_cast<uint32_t>(p.band_m / CM);
    const uint32_t band_size = band_units * nt32;
    const uint32_t band = u32 / band_size;
    const uint32_t within = u32 - band * band_size;
    const uint32_t in_band =
        static_cast<uint32_t>(::min(static_cast<int64_t>(band_units), m_units - band * band_units));
    const uint32_t n_blk32 = within / in_band;
    const int64_t n_blk = n_blk32;
    const int64_t mu = static_cast<int64_t>(band) * band_units + (within - n_blk32 * in_band);
    const int64_t m_blk = mu * CM + rank;
    ti.m0 = m_blk * kTileM;
    ti.y_row0 = ti.m0;
    ti.m_end = p.m;
    ti.sfa_unit = m_blk < m_tiles ? m_blk * a_tiles_k : -1;
    ti.sfa_rt = static_cast<int32_t>(m_blk);
    ti.sfa_kt0 = 0;
    ti.n0 = n_blk * BN;
    ti.b_row0 = ti.n0;
    ti.sfb_rt = static_cast<int32_t>(ti.n0 / 128);
    ti.sfb_kt0 = 0;
    ti.sfb_unit = ti.sfb_rt * b_tiles_k;
  }
  return ti;
}

}  // namespace mx
