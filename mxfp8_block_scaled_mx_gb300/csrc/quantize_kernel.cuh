// quantize_kernel.cuh -- the MX quantization kernel (bf16 or FP32 ->
// E4M3 / E5M2 / E2M3 / E3M2 / E2M1 codes plus E8M0 block scales in the
// swizzled tensor-core layout), shared by the translation units that
// instantiate it for each input type.
//
// "Low-Precision GPU Programming" (leetllm.com): section "Microscaling: the
// two-row experiment" (32-element blocks, one E8M0 power-of-two scale per
// block, both orientations from the original wide data) and section
// "Numerical hazards: subnormals, saturation, and rounding" (round to
// nearest even, subnormals kept, saturation after rounding).
//
// The kernel is HBM-bound (stochastic rounding of both orientations from
// one read comes closest to being compute-bound), so it is built
// around deep prefetch: one persistent block per SM, a producer thread that
// streams tiles of x (128 rows of 128 bf16 or FP32 columns, 32 or 64 KB;
// 64 FP32 columns when columnwise codes are written too) into a ring of
// shared-memory slots with cp.async.bulk.tensor, and groups of eight
// consumer warps that take tiles round-robin, straight out of shared memory
// while the next tiles are in flight.
//  - Rowwise (bf16): the thread that holds one 32-element block reduces its
//    amax with SIMD max.u16x2 on the bf16 bit patterns, derives the scale
//    exponent from the bit pattern, scales by an exact power of two and
//    converts pairs with the hardware cvt.rn.satfinite instruction.  The
//    tile's 128 x 4 scales form exactly one 512-byte swizzled unit,
//    assembled in shared memory and written with one coalesced store.
//  - Columnwise (bf16): each thread reduces and encodes two adjacent
//    columns of a 32-row block (one 32-bit shared load and one SIMD max per
//    row), the codes are transposed in shared memory and written back as
//    128-byte rows of the [cols, rows] output, again with one 512-byte scale
//    unit per tile.
//  - FP32 input: a rowwise-only pass takes 128-column tiles (64 KB slots,
//    two blocks a thread, one after the other); with columnwise codes the
//    tiles hold 64 columns in 32 KB, each thread takes one block (rowwise)
//    or one column block (columnwise), and a tile fills half of each
//    512-byte scale unit (the half is written in place, the whole unit when
//    the tile is the matrix's last).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "groups.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "status.cuh"

namespace mx {
namespace {

constexpr int kTile = 128;                    // rows of x per tile (and bf16 columns)
constexpr int kGroupThreads = 256;            // one consumer group: 8 warps
constexpr int kTileBytes = kTile * kTile * 2; // 32 KB: 128 rows of 256 bytes

// Columns of x per tile: 128 bf16 (32 KB); FP32 128 (64 KB) for a
// rowwise-only pass and 64 (32 KB, half of each scale unit) when the
// columnwise codes are written too.
template <bool F32, bool COL>
constexpr int kTileCols = (F32 && COL) ? 64 : 128;
constexpr int kColPitch = 144;                // bytes per transposed code row in smem

// Per-halfword unsigned max of two packed pairs (one SIMD instruction).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Element formats (library enum order): 0 E4M3, 1 E5M2, 2 E2M3, 3 E3M2,
// 4 E2M1.  kEmax = exponent of the largest binade; the largest finite value
// has significand kMaxNum / kMaxDen (1.75 for E4M3, E5M2 and E3M2, 1.875 for
// E2M3, 1.5 for E2M1); kBits = code width.
template <int FMT>
struct ElemFmt {
  static constexpr int kEmax = FMT == 0 ? 8 : FMT == 1 ? 15 : FMT == 3 ? 4 : 2;
  static constexpr uint32_t kMaxNum = FMT == 2 ? 15u : FMT == 4 ? 3u : 7u;
  static constexpr uint32_t kMaxDen = FMT == 2 ? 8u : FMT == 4 ? 2u : 4u;
  static constexpr int kBits = FMT <= 1 ? 8 : FMT == 4 ? 4 : 6;
  // code written for every element of a NaN/Inf block (4 codes per word
  // for FP8; the narrower formats have no NaN code and write 0)
  static constexpr uint32_t kNanWord = FMT <= 1 ? 0x7F7F7F7Fu : 0u;
};

// Scale exponent e of a block with finite amax (bit pattern `a` of a bf16,
// or of an FP32 with F32): floor rule e = floor(log2 amax) - emax_elem; the
// ceil rule adds one when the significand of amax exceeds that of the
// format's maximum.  amax = 0 gives e = 0 (S = 1).  Clamped to [-127, 127].
template <int FMT, bool F32 = false>
__device__ __forceinline__ int scale_exponent(uint32_t a, int rule) {
  using F = ElemFmt<FMT>;
  constexpr int kM = F32 ? 23 : 7;          // stored significand bits of the input
  constexpr int kSubExp = F32 ? 149 : 133;  // a subnormal input is mant * 2^-kSubExp
  if (a == 0) return 0;
  const uint32_t ef = a >> kM;
  const uint32_t mant = a & ((1u << kM) - 1u);
  int fl;
  bool above;
  if (ef != 0) {
    fl = static_cast<int>(ef) - 127;
    // (1 + mant / 2^kM) > max significand
    above = F::kMaxDen * ((1u << kM) + mant) > (F::kMaxNum << kM);
  } else {
    const int p = 31 - __clz(mant);
    fl = p - kSubExp;
    above = F::kMaxDen * mant > (F::kMaxNum << p);
  }
  int e = fl - F::kEmax + ((rule == 1 && above) ? 1 : 0);
  return min(max(e, -127), 127);
}

// 2^-e as a float (exact: e in [-127, 127] keeps the exponent normal).
__device__ __forceinline__ float pow2_neg(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// Two floats -> two codes, RNE with saturation to the finite range; `lo`
// lands in the low part.  FP8 and FP6: one code per byte (16 bits; a 6-bit
// code in the low bits of its byte); FP4: one code per nibble (8 bits).
template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
  if constexpr (FMT == 4) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
  } else {
    uint16_t r;
    if constexpr (FMT == 0) {
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    } else if constexpr (FMT == 1) {
      asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    } else if constexpr (FMT == 2) {
      asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    } else {
      asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    }
    return r;
  }
}

// Four 6-bit codes, one per byte of w, packed into 24 bits (code i at bits
// [6i, 6i + 6)).
__device__ __forceinline__ uint32_t pack4_fp6(uint32_t w) {
  return (w & 0x3Fu) | ((w >> 8) & 0x3Fu) << 6 | ((w >> 16) & 0x3Fu) << 12 |
         ((w >> 24) & 0x3Fu) << 18;
}

// Sixteen 6-bit codes (one per byte of w0..w3) -> one 16-byte container:
// the 96 packed bits, then four zero bytes.
__device__ __forceinline__ uint4 container16_fp6(uint32_t w0, uint32_t w1, uint32_t w2,
                                                 uint32_t w3) {
  const uint32_t g0 = pack4_fp6(w0), g1 = pack4_fp6(w1), g2 = pack4_fp6(w2), g3 = pack4_fp6(w3);
  return make_uint4(g0 | g1 << 24, g1 >> 8 | g2 << 16, g2 >> 16 | g3 << 8, 0u);
}

// The two bf16 of a word (low half first) as FP32, each times its own
// power-of-two factor, in one packed FP32x2 multiply.  The products are
// exact (an 8-bit significand times a power of two, far from the FP32
// range limits), so they equal the scalar products bit for bit.
__device__ __forceinline__ float2 scale_pair(uint32_t w, float m_lo, float m_hi) {
  uint64_t x, m, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(w << 16), "r"(w & 0xFFFF0000u));
  asm("mov.b64 %0, {%1, %2};" : "=l"(m) : "f"(m_lo), "f"(m_hi));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(m));
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}

// Two bf16 packed in a word -> two codes (16 bits), after an exact scaling.
template <int FMT>
__device__ __forceinline__ uint32_t encode_word(uint32_t w, float mul) {
  const float2 v = scale_pair(w, mul, mul);
  return cvt_pair<FMT>(v.x, v.y);
}

// Eight bf16 -> eight codes: FP8 and FP6 one per byte (x: codes 0-3,
// y: codes 4-7); FP4 packed in x (code i in bits [4i, 4i + 4)), y = 0.
template <int FMT>
__device__ __forceinline__ uint2 encode8(const uint4 v, float mul) {
  uint2 r;
  if constexpr (FMT == 4) {
    r.x = encode_word<FMT>(v.x, mul) | (encode_word<FMT>(v.y, mul) << 8) |
          (encode_word<FMT>(v.z, mul) << 16) | (encode_word<FMT>(v.w, mul) << 24);
    r.y = 0u;
  } else {
    r.x = encode_word<FMT>(v.x, mul) | (encode_word<FMT>(v.y, mul) << 16);
    r.y = encode_word<FMT>(v.z, mul) | (encode_word<FMT>(v.w, mul) << 16);
  }
  return r;
}

// Two FP32 (bit patterns lo, hi) times their power-of-two factors, in one
// packed FP32x2 multiply.  The products are exact except below 2^-126,
// where the multiply may round; every such value is under 2^-16 of the
// smallest step of any of the formats, so round to nearest even (and
// stochastic rounding with 16-bit draws) takes it to zero, of its sign,
// exactly as it would the exact product.
__device__ __forceinline__ float2 scale_f32_pair(uint32_t lo, uint32_t hi, float m_lo, float m_hi) {
  uint64_t x, m, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(lo), "r"(hi));
  asm("mov.b64 %0, {%1, %2};" : "=l"(m) : "f"(m_lo), "f"(m_hi));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(m));
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}

// Eight FP32 (a: elements 0-3, b: elements 4-7) -> eight codes, laid out as
// encode8.
template <int FMT>
__device__ __forceinline__ uint2 encode8_f32(const uint4 a, const uint4 b, float mul) {
  const float2 s0 = scale_f32_pair(a.x, a.y, mul, mul), s1 = scale_f32_pair(a.z, a.w, mul, mul);
  const float2 s2 = scale_f32_pair(b.x, b.y, mul, mul), s3 = scale_f32_pair(b.z, b.w, mul, mul);
  const uint32_t p0 = cvt_pair<FMT>(s0.x, s0.y), p1 = cvt_pair<FMT>(s1.x, s1.y);
  const uint32_t p2 = cvt_pair<FMT>(s2.x, s2.y), p3 = cvt_pair<FMT>(s3.x, s3.y);
  if constexpr (FMT == 4) return make_uint2(p0 | p1 << 8 | p2 << 16 | p3 << 24, 0u);
  return make_uint2(p0 | p1 << 16, p2 | p3 << 16);
}

// Stochastic rounding of two exactly scaled values onto the format grid
// (section "Rounding: RNE versus stochastic rounding"), r holding v.x's
// 16-bit random integer in its low half and v.y's in its high half: with
// l <= |v| < u neighbouring grid values, |v| goes to u iff its random
// integer is below floor(frac * 2^16), frac = (|v| - l) / (u - l).  Each
// result is a grid value (or one step past the maximum, which the
// saturating conversion then clamps), with the sign of v.  v is exact (a
// bf16 or an FP32 times a power of two; an FP32 product below 2^-126 goes
// to zero either way).
template <int FMT>
__device__ __forceinline__ float2 sr_to_grid2(float2 v, uint32_t r) {
  // significand bits and smallest normal exponent: E4M3 3 / -6, E5M2 2 /
  // -14, E2M3 3 / 0, E3M2 2 / -2, E2M1 1 / 0
  constexpr int kMantBits = (FMT == 0 || FMT == 2) ? 3 : FMT == 4 ? 1 : 2;
  constexpr int kMinNormalExp = FMT == 0 ? -6 : FMT == 1 ? -14 : FMT == 3 ? -2 : 0;
  constexpr int kDrop = 23 - kMantBits;  // FP32 significand bits below the format's grid
  // v * 2^-kShift takes the format's smallest normal m = 2^kMinNormalExp
  // to FP32's (2^-126).  Above it the FP32 pattern keeps the format's
  // significand bits over kDrop dropped bits; below it the pattern is an
  // FP32 subnormal, linear in the value, whose unit 2^-149 makes the
  // format's subnormal quantum exactly 2^kDrop units: in both ranges l is
  // the pattern with the low kDrop bits cleared and u is l plus one step (a
  // carry into the exponent gives the next binade's first value, or m).
  // The top 16 dropped bits are floor(frac * 2^16) (the multiply rounds
  // toward zero, which only clears bits below them), and adding 0xFFFF - r
  // to them carries into the kept bits exactly when r < floor(frac * 2^16)
  // (the bits below them are too few to carry), so u or l is the sum with
  // the dropped bits cleared.  The sign bit rides along (signed zeros
  // included), and the scaling back by 2^kShift is exact.  Both multiplies
  // work on the pair at once (FP32x2).
  constexpr int kShift = kMinNormalExp + 126;
  constexpr uint32_t kMask = ~((1u << kDrop) - 1u);
  const float down = __uint_as_float(static_cast<uint32_t>(127 - kShift) << 23);
  const float up = __uint_as_float(static_cast<uint32_t>(127 + kShift) << 23);
  uint64_t x, m, p;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(v.x), "f"(v.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(m) : "f"(down), "f"(down));
  asm("mul.rz.f32x2 %0, %1, %2;" : "=l"(p) : "l"(x), "l"(m));
  uint32_t b0, b1;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(b0), "=r"(b1) : "l"(p));
  const uint32_t nr = ~r;  // 0xFFFF - r in each half
  const uint32_t t0 = (b0 + ((nr & 0xFFFFu) << (kDrop - 16))) & kMask;
  const uint32_t t1 = (b1 + ((nr >> 16) << (kDrop - 16))) & kMask;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(t0), "r"(t1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(m) : "f"(up), "f"(up));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(x), "l"(m));
  float2 g;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(g.x), "=f"(g.y) : "l"(p));
  return g;
}

// Two bf16 of a word with their two 16-bit random integers -> two codes.
template <int FMT>
__device__ __forceinline__ uint32_t encode_word_sr(uint32_t w, uint32_t r, float mul) {
  const float2 g = sr_to_grid2<FMT>(scale_pair(w, mul, mul), r);
  return cvt_pair<FMT>(g.x, g.y);
}

// Eight bf16 with their random integers -> eight codes, laid out as encode8.
template <int FMT>
__device__ __forceinline__ uint2 encode8_sr(const uint4 v, const uint4 r, float mul) {
  uint2 q;
  if constexpr (FMT == 4) {
    q.x = encode_word_sr<FMT>(v.x, r.x, mul) | (encode_word_sr<FMT>(v.y, r.y, mul) << 8) |
          (encode_word_sr<FMT>(v.z, r.z, mul) << 16) | (encode_word_sr<FMT>(v.w, r.w, mul) << 24);
    q.y = 0u;
  } else {
    q.x = encode_word_sr<FMT>(v.x, r.x, mul) | (encode_word_sr<FMT>(v.y, r.y, mul) << 16);
    q.y = encode_word_sr<FMT>(v.z, r.z, mul) | (encode_word_sr<FMT>(v.w, r.w, mul) << 16);
  }
  return q;
}

// Two FP32 (bit patterns lo, hi) with their two 16-bit random integers (r:
// lo's in the low half) -> two codes.
template <int FMT>
__device__ __forceinline__ uint32_t encode_f32_pair_sr(uint32_t lo, uint32_t hi, uint32_t r,
                                                       float mul) {
  const float2 g = sr_to_grid2<FMT>(scale_f32_pair(lo, hi, mul, mul), r);
  return cvt_pair<FMT>(g.x, g.y);
}

// Eight FP32 with their random integers (r: two per word, element order)
// -> eight codes, laid out as encode8.
template <int FMT>
__device__ __forceinline__ uint2 encode8_f32_sr(const uint4 a, const uint4 b, const uint4 r,
                                                float mul) {
  const uint32_t p0 = encode_f32_pair_sr<FMT>(a.x, a.y, r.x, mul);
  const uint32_t p1 = encode_f32_pair_sr<FMT>(a.z, a.w, r.y, mul);
  const uint32_t p2 = encode_f32_pair_sr<FMT>(b.x, b.y, r.z, mul);
  const uint32_t p3 = encode_f32_pair_sr<FMT>(b.z, b.w, r.w, mul);
  if constexpr (FMT == 4) return make_uint2(p0 | p1 << 8 | p2 << 16 | p3 << 24, 0u);
  return make_uint2(p0 | p1 << 16, p2 | p3 << 16);
}

constexpr uint8_t kNanScale = 0xFF;

// Byte offset of (local row r, local block c) inside a 512-byte scale unit.
__device__ __forceinline__ int unit_offset(int r, int c) {
  return (r & 31) * 16 + (r >> 5) * 4 + c;
}

// Offset in a ring slot of byte `byte` (0..255) of tile row r.  The tensor
// copy writes the 128 x 128 bf16 tile as two 64-column halves of 128 rows x
// 128 bytes with the 128-byte swizzle: 16-byte chunk c of row r lands at
// chunk c ^ (r % 8) of its row.  Then a warp reading one 64-byte block from
// each of eight rows (rowwise) or one 128-byte row segment (columnwise)
// touches every shared-memory bank the same number of times.
__device__ __forceinline__ int tile_offset(int r, int byte) {
  return (byte >> 7) * (kTile * 128) + r * 128 + ((((byte >> 4) & 7) ^ (r & 7)) << 4) + (byte & 15);
}

// Largest magnitude bit pattern (sign cleared) among the 32 bf16 of v.  For
// non-NaN bf16 the unsigned order of these patterns is the order of |x|;
// NaN patterns sort above +Inf (0x7F80).
__device__ __forceinline__ uint32_t amax_bits32(const uint4 (&v)[4]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    m = max_u16x2(m, max_u16x2(v[j].x & 0x7FFF7FFFu, v[j].y & 0x7FFF7FFFu));
    m = max_u16x2(m, max_u16x2(v[j].z & 0x7FFF7FFFu, v[j].w & 0x7FFF7FFFu));
  }
  return max(m & 0xFFFFu, m >> 16);
}

// Largest magnitude bit pattern (sign cleared) among the 32 FP32 of v; as
// for bf16, NaN patterns sort above +Inf (0x7F800000).
__device__ __forceinline__ uint32_t amax_bits32_f32(const uint4 (&v)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    m = max(m, max(max(v[j].x & 0x7FFFFFFFu, v[j].y & 0x7FFFFFFFu),
                   max(v[j].z & 0x7FFFFFFFu, v[j].w & 0x7FFFFFFFu)));
  }
  return m;
}

struct Tile {
  int64_t x_row0;       // first row of x in the tile
  int64_t c0;           // first column of x in the tile
  int64_t rows_valid;   // rows of the tile that exist (<= 128)
  int64_t scale_rt;     // row-tile index of the rowwise scale unit
};

struct GroupInfo {
  int32_t off[kMaxGroups + 1];
  int32_t tiles[kMaxGroups + 1];
  int32_t valid;
};

// Tile t of the launch (kCols columns of x wide): dense tiles are (row
// tile, column tile) in row-major order; grouped tiles walk the per-group padded row tiles.  The
// grouped columnwise pass divides in 32 bits and finds the tile's group by
// walking forward from the previous tile's group (`g_hint`, per caller: its
// tiles come in increasing order) instead of a binary search: 11 % faster
// there, while the walk measured slower on the rowwise pass, which keeps
// the search.  Dense single-orientation passes divide in 32 bits too (1-2 %
// faster; the two-orientation pass measured slower that way).  The host
// keeps those launches' tile counts below 2^32.
template <bool GROUPED, bool ROW, bool COL, int kCols>
__device__ __forceinline__ Tile tile_of(const QuantizeParams& p, int64_t t, int64_t col_tiles,
                                        const GroupInfo* gi, int& g_hint) {
  Tile tl;
  int64_t rt;
  if constexpr ((GROUPED && COL) || (!GROUPED && ROW != COL))
    rt = static_cast<uint32_t>(t) / static_cast<uint32_t>(col_tiles);
  else
    rt = t / col_tiles;
  tl.c0 = (t - rt * col_tiles) * kCols;
  tl.scale_rt = rt;
  if constexpr (GROUPED) {
    int g;
    if constexpr (COL) {
      g = g_hint;
      while (g + 1 < p.groups && gi->tiles[g + 1] <= rt) ++g;
      g_hint = g;
    } else {
      g = find_group(gi->tiles, p.groups, static_cast<int32_t>(rt));
    }
    tl.x_row0 = static_cast<int64_t>(gi->off[g]) + (rt - gi->tiles[g]) * kTile;
    tl.rows_valid = ::min(static_cast<int64_t>(kTile), gi->off[g + 1] - tl.x_row0);
  } else {
    tl.x_row0 = rt * kTile;
    tl.rows_valid = ::min(static_cast<int64_t>(kTile), p.rows - tl.x_row0);
  }
  return tl;
}

__device__ __forceinline__ void group_bar(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(kGroupThreads) : "memory");
}

// Group barrier that also returns, to every thread, whether `pred` held for
// any thread of the group (so a bail-out decision is uniform).
__device__ __forceinline__ bool group_bar_any(int group, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(1 + group), "r"(kGroupThreads)
      : "memory");
  return r != 0;
}

// One block's 32 codes (c[j]: codes 8j..8j+7, laid out as encode8 gives
// them) into the code row at `rowp`, starting at element column gcb: FP8 32
// bytes; FP6 / FP4 one 16-byte container per 16-element run; packed
// storage 16 (FP4) or 24 (FP6) bytes.  With `half` (a partial final block
// of 16 elements; not in packed storage) only the first run is stored.
template <int FMT, bool PACKED>
__device__ __forceinline__ void store_row_block(uint8_t* rowp, int64_t gcb, const uint2 (&c)[4],
                                                bool half) {
  using F = ElemFmt<FMT>;
  if constexpr (F::kBits == 8) {
    *reinterpret_cast<uint4*>(rowp + gcb) = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
    if (!half)
      *reinterpret_cast<uint4*>(rowp + gcb + 16) = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
  } else if constexpr (F::kBits == 4) {
    // eight codes per 32-bit word (code i in bits [4i, 4i + 4))
    if constexpr (PACKED) {
      *reinterpret_cast<uint4*>(rowp + gcb / 2) = make_uint4(c[0].x, c[1].x, c[2].x, c[3].x);
    } else {  // two 16-element runs, each 8 bytes of codes then 8 zero bytes
      *reinterpret_cast<uint4*>(rowp + gcb) = make_uint4(c[0].x, c[1].x, 0u, 0u);
      if (!half) *reinterpret_cast<uint4*>(rowp + gcb + 16) = make_uint4(c[2].x, c[3].x, 0u, 0u);
    }
  } else {
    // 6-bit codes: each run of 16 is 96 packed bits (12 bytes)
    uint32_t g[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      g[2 * j] = pack4_fp6(c[j].x);
      g[2 * j + 1] = pack4_fp6(c[j].y);
    }
    const uint32_t w0 = g[0] | g[1] << 24, w1 = g[1] >> 8 | g[2] << 16, w2 = g[2] >> 16 | g[3] << 8;
    const uint32_t w3 = g[4] | g[5] << 24, w4 = g[5] >> 8 | g[6] << 16, w5 = g[6] >> 16 | g[7] << 8;
    if constexpr (PACKED) {
      uint2* d = reinterpret_cast<uint2*>(rowp + gcb * 3 / 4);
      d[0] = make_uint2(w0, w1);
      d[1] = make_uint2(w2, w3);
      d[2] = make_uint2(w4, w5);
    } else {  // each run's 12 bytes, then 4 zero bytes
      *reinterpret_cast<uint4*>(rowp + gcb) = make_uint4(w0, w1, w2, 0u);
      if (!half) *reinterpret_cast<uint4*>(rowp + gcb + 16) = make_uint4(w3, w4, w5, 0u);
    }
  }
}

// One column block's 32 codes (q[i]: those of rows 4i..4i+3, FP8 / FP6 one
// per byte, FP4 one per nibble) into transposed row c of the tile's code
// buffer, block rb: FP8 32 bytes; FP6 / FP4 one 16-byte container per run;
// packed storage 16 (FP4) or 24 (FP6) bytes.
template <int FMT, bool PACKED>
__device__ __forceinline__ void stage_col_block(uint8_t* s_q, int c, int rb, const uint32_t (&q)[8]) {
  using F = ElemFmt<FMT>;
  uint8_t* row = s_q + c * kColPitch;
  if constexpr (PACKED && F::kBits == 4) {
    *reinterpret_cast<uint4*>(row + rb * 16) = make_uint4(
        q[0] | q[1] << 16, q[2] | q[3] << 16, q[4] | q[5] << 16, q[6] | q[7] << 16);
  } else if constexpr (PACKED) {
    // eight groups of four 6-bit codes, 24 bits each, in 24 bytes
    uint2* e = reinterpret_cast<uint2*>(row + rb * 24);
    uint32_t g[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = pack4_fp6(q[i]);
    e[0] = make_uint2(g[0] | g[1] << 24, g[1] >> 8 | g[2] << 16);
    e[1] = make_uint2(g[2] >> 16 | g[3] << 8, g[4] | g[5] << 24);
    e[2] = make_uint2(g[5] >> 8 | g[6] << 16, g[6] >> 16 | g[7] << 8);
  } else if constexpr (F::kBits == 8) {
    uint4* d = reinterpret_cast<uint4*>(row + rb * 32);
    d[0] = make_uint4(q[0], q[1], q[2], q[3]);
    d[1] = make_uint4(q[4], q[5], q[6], q[7]);
  } else if constexpr (F::kBits == 6) {
    uint4* d = reinterpret_cast<uint4*>(row + rb * 32);
    d[0] = container16_fp6(q[0], q[1], q[2], q[3]);
    d[1] = container16_fp6(q[4], q[5], q[6], q[7]);
  } else {
    uint4* d = reinterpret_cast<uint4*>(row + rb * 32);
    d[0] = make_uint4(q[0] | q[1] << 16, q[2] | q[3] << 16, 0u, 0u);
    d[1] = make_uint4(q[4] | q[5] << 16, q[6] | q[7] << 16, 0u, 0u);
  }
}

// One consumer group quantizes one tile held in ring slot `xs` (128 rows of
// 256 bytes: 128 bf16 or, with F32, 64 FP32 columns); with SR, `rs` holds
// the tile's 16-bit random integers in the bf16 tile layout (the first 128
// bytes of each row with F32).  `lt` is the thread's index inside the
// group.  Grouped columnwise tiles may hold rows of the next group past
// rows_valid: those rows count as zeros (the zero-padded final block of the
// group), and the tile's full 128 transposed columns are written, padding
// included.  An FP32 tile covers half of each 512-byte scale unit: unit
// columns 2h, 2h + 1 (rowwise) or unit rows [64h, 64h + 64) (columnwise),
// h = (c0 / 64) % 2.
template <int FMT, bool ROW, bool COL, bool GROUPED, bool SR, bool PACKED, bool F32>
__device__ __forceinline__ void quantize_tile(const QuantizeParams& p, const Tile& tl,
                                              const uint8_t* xs, const uint8_t* rs, uint8_t* s_q,
                                              uint8_t* s_unit_row, uint8_t* s_unit_col,
                                              uint64_t* empty_bar, int group, int lt) {
  using F = ElemFmt<FMT>;
  constexpr int kCols = kTileCols<F32, COL>;
  const uint32_t lane = lt & 31;
  const int half = static_cast<int>(tl.c0 >> 6) & 1;  // FP32: which half of the scale units
  // bytes per code row: one per element, or w / 8 in packed storage
  const int64_t row_bytes = PACKED ? p.cols * F::kBits / 8 : p.cols;

  if constexpr (ROW && F32 && kCols == 128) {
    // 128 FP32 columns, four blocks a row: thread lt quantizes blocks
    // lt / 128 and lt / 128 + 2 of tile row lt % 128, one after the other
    // (a warp reads 32 consecutive rows, conflict-free under the swizzle).
    const int lr = lt & 127;
    // not unrolled: the second block's loads would be hoisted above the
    // first block's work and spill with stochastic rounding
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
      const int bq = (lt >> 7) + 2 * j;
      const int64_t gcb = tl.c0 + bq * 32;
      const bool blk_ok = gcb < p.cols;
      uint4 v[8];
      uint4 rv[SR ? 4 : 1];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        v[i] = *reinterpret_cast<const uint4*>(xs + tile_offset(lr, bq * 128 + i * 16));
      if constexpr (SR) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          rv[i] = *reinterpret_cast<const uint4*>(rs + tile_offset(lr, bq * 64 + i * 16));
      }
      if (j == 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar);  // slot fully read by this warp
      }
      uint2 c[4];
      uint8_t sbyte;
      const uint32_t a = amax_bits32_f32(v);
      if (a >= 0x7F800000u) {  // NaN or Inf in the block
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = make_uint2(F::kNanWord, F::kNanWord);
        sbyte = kNanScale;
      } else {
        const int e = scale_exponent<FMT, true>(a, p.rule);
        const float mul = pow2_neg(e);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if constexpr (SR) {
            c[i] = encode8_f32_sr<FMT>(v[2 * i], v[2 * i + 1], rv[SR ? i : 0], mul);
          } else {
            c[i] = encode8_f32<FMT>(v[2 * i], v[2 * i + 1], mul);
          }
        }
        sbyte = static_cast<uint8_t>(e + 127);
      }
      if (blk_ok && lr < tl.rows_valid) {
        store_row_block<FMT, PACKED>(p.q_row + (tl.x_row0 + lr) * row_bytes, gcb, c,
                                     gcb + 16 >= p.cols);
        s_unit_row[unit_offset(lr, bq)] = sbyte;
      }
    }
  } else if constexpr (ROW && F32) {
    // Thread lt quantizes block lt / 128 (of the tile's two) of tile row
    // lt % 128; a warp reads 32 consecutive rows, conflict-free under the
    // swizzle.
    const int lr = lt & 127;
    const int bq = lt >> 7;
    const int64_t gcb = tl.c0 + bq * 32;  // first column of the block
    // cols % 16 == 0: a block is whole, absent, or a final block of 16
    // columns (the tensor copy filled the rest with zeros)
    const bool blk_ok = gcb < p.cols;
    uint4 v[8];
    uint4 rv[SR ? 4 : 1];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const uint4*>(xs + tile_offset(lr, bq * 128 + j * 16));
    if constexpr (SR) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        rv[j] = *reinterpret_cast<const uint4*>(rs + tile_offset(lr, bq * 64 + j * 16));
    }
    if constexpr (!COL) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);  // slot fully read by this warp
    }
    uint2 c[4];
    uint8_t sbyte;
    const uint32_t a = amax_bits32_f32(v);
    if (a >= 0x7F800000u) {  // NaN or Inf in the block
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = make_uint2(F::kNanWord, F::kNanWord);
      sbyte = kNanScale;
    } else {
      const int e = scale_exponent<FMT, true>(a, p.rule);
      const float mul = pow2_neg(e);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (SR) {
          c[j] = encode8_f32_sr<FMT>(v[2 * j], v[2 * j + 1], rv[SR ? j : 0], mul);
        } else {
          c[j] = encode8_f32<FMT>(v[2 * j], v[2 * j + 1], mul);
        }
      }
      sbyte = static_cast<uint8_t>(e + 127);
    }
    if (blk_ok && lr < tl.rows_valid) {
      store_row_block<FMT, PACKED>(p.q_row + (tl.x_row0 + lr) * row_bytes, gcb, c,
                                   gcb + 16 >= p.cols);
      s_unit_row[unit_offset(lr, 2 * half + bq)] = sbyte;
    }
  } else if constexpr (ROW && SR && !COL) {
    // Rowwise-only stochastic rounding: the same blocks as below, the
    // thread's two rows one after the other, so that only one row's values
    // and draws (32 registers) are live at a time; loading both rows first
    // spilled and ran 3 % slower.
    const int bq = lt & 3;
    const int lr0 = lt >> 2;
    const int64_t gcb = tl.c0 + bq * 32;
    const bool blk_ok = gcb < p.cols;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      const int lr = lr0 + 64 * h;
      uint4 v[4], rv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int off = tile_offset(lr, bq * 64 + j * 16);
        v[j] = *reinterpret_cast<const uint4*>(xs + off);
        rv[j] = *reinterpret_cast<const uint4*>(rs + off);
      }
      if (h == 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar);  // slot fully read by this warp
      }
      uint2 c[4];
      uint8_t sbyte;
      const uint32_t a = amax_bits32(v);
      if (a >= 0x7F80u) {
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = make_uint2(F::kNanWord, F::kNanWord);
        sbyte = kNanScale;
      } else {
        const int e = scale_exponent<FMT>(a, p.rule);
        const float mul = pow2_neg(e);
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = encode8_sr<FMT>(v[j], rv[j], mul);
        sbyte = static_cast<uint8_t>(e + 127);
      }
      if (blk_ok && lr < tl.rows_valid) {
        store_row_block<FMT, PACKED>(p.q_row + (tl.x_row0 + lr) * row_bytes, gcb, c,
                                     gcb + 16 >= p.cols);
        s_unit_row[unit_offset(lr, bq)] = sbyte;
      }
    }
  } else if constexpr (ROW) {
    // Thread lt quantizes the 32-element block lt % 4 of tile rows lt / 4
    // and lt / 4 + 64: it holds the whole block, so the amax needs no
    // shuffles and the scale exponent is derived once per block.
    const int bq = lt & 3;
    const int lr0 = lt >> 2;
    const int64_t gcb = tl.c0 + bq * 32;  // first column of the block
    // cols % 16 == 0: a block is whole, absent, or a final block of 16
    // columns (the tensor copy filled the rest with zeros)
    const bool blk_ok = gcb < p.cols;
    uint4 v[2][4];
    uint4 rv[SR ? 2 : 1][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int off = tile_offset(lr0 + 64 * h, bq * 64 + j * 16);
        v[h][j] = *reinterpret_cast<const uint4*>(xs + off);
        if constexpr (SR) rv[h][j] = *reinterpret_cast<const uint4*>(rs + off);
      }
    }
    if constexpr (!COL) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);  // slot fully read by this warp
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int lr = lr0 + 64 * h;
      uint2 c[4];
      uint8_t sbyte;
      const uint32_t a = amax_bits32(v[h]);
      if (a >= 0x7F80u) {  // NaN or Inf in the block
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = make_uint2(F::kNanWord, F::kNanWord);
        sbyte = kNanScale;
      } else {
        const int e = scale_exponent<FMT>(a, p.rule);
        const float mul = pow2_neg(e);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (SR) {
            c[j] = encode8_sr<FMT>(v[h][j], rv[SR ? h : 0][j], mul);
          } else {
            c[j] = encode8<FMT>(v[h][j], mul);
          }
        }
        sbyte = static_cast<uint8_t>(e + 127);
      }
      if (!blk_ok || lr >= tl.rows_valid) continue;
      store_row_block<FMT, PACKED>(p.q_row + (tl.x_row0 + lr) * row_bytes, gcb, c,
                                   gcb + 16 >= p.cols);
      s_unit_row[unit_offset(lr, bq)] = sbyte;
    }
  }

  if constexpr (COL && F32) {
    // Thread lt: column lt % 64 of the tile, 32-row block lt / 64; a warp
    // reads one 128-byte row segment per row, conflict-free.
    const int cl = lt & 63;
    const int rb = lt >> 6;
    const bool ok = tl.c0 + cl < p.cols && rb * 32 < tl.rows_valid;
    uint32_t w[32];
    uint32_t rw[SR ? 32 : 1];
    uint32_t a = 0;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      w[r] = *reinterpret_cast<const uint32_t*>(xs + tile_offset(rb * 32 + r, cl * 4));
      if constexpr (SR) rw[r] = *reinterpret_cast<const uint16_t*>(rs + tile_offset(rb * 32 + r, cl * 2));
    }
    if constexpr (GROUPED) {
      // rows of the next group in a partial block count as zeros (uniform
      // across the warp: one 32-row block per warp)
      if (rb * 32 + 32 > tl.rows_valid) {
#pragma unroll
        for (int r = 0; r < 32; ++r)
          if (rb * 32 + r >= tl.rows_valid) w[r] = 0u;
      }
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) a = max(a, w[r] & 0x7FFFFFFFu);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar);  // slot fully read by this warp
    const bool nan = a >= 0x7F800000u;
    const int e = nan ? 0 : scale_exponent<FMT, true>(a, p.rule);
    const float m = pow2_neg(e);
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // rows 4i..4i+3 of the column
      uint32_t p01, p23;
      if constexpr (SR) {
        p01 = encode_f32_pair_sr<FMT>(w[4 * i], w[4 * i + 1], rw[4 * i] | rw[4 * i + 1] << 16, m);
        p23 = encode_f32_pair_sr<FMT>(w[4 * i + 2], w[4 * i + 3], rw[4 * i + 2] | rw[4 * i + 3] << 16, m);
      } else {
        const float2 s01 = scale_f32_pair(w[4 * i], w[4 * i + 1], m, m);
        const float2 s23 = scale_f32_pair(w[4 * i + 2], w[4 * i + 3], m, m);
        p01 = cvt_pair<FMT>(s01.x, s01.y);
        p23 = cvt_pair<FMT>(s23.x, s23.y);
      }
      q[i] = nan ? F::kNanWord : (p01 | p23 << (FMT == 4 ? 8 : 16));
    }
    stage_col_block<FMT, PACKED>(s_q, cl, rb, q);
    if (ok) s_unit_col[unit_offset(64 * half + cl, rb)] = nan ? kNanScale : static_cast<uint8_t>(e + 127);
  } else if constexpr (COL) {
    // Thread lt: columns 2*(lt % 64) and 2*(lt % 64) + 1, 32-row block
    // lt / 64.  One 32-bit shared load gives both columns of a row, so the
    // amax of the two column blocks is one SIMD max per row.
    const int cp = lt & 63;
    const int rb = lt >> 6;
    const bool ok = tl.c0 + 2 * cp < p.cols && rb * 32 < tl.rows_valid;
    uint32_t w[32];
    uint32_t rw[SR ? 32 : 1];
    uint32_t a2 = 0;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const int off = tile_offset(rb * 32 + r, cp * 4);
      w[r] = *reinterpret_cast<const uint32_t*>(xs + off);
      if constexpr (SR) rw[r] = *reinterpret_cast<const uint32_t*>(rs + off);
    }
    if constexpr (GROUPED) {
      // rows of the next group in a partial block count as zeros (uniform
      // across the warp: one 32-row block per warp); testing every row of
      // every block cost the grouped columnwise pass 11 % of its time
      if (rb * 32 + 32 > tl.rows_valid) {
#pragma unroll
        for (int r = 0; r < 32; ++r)
          if (rb * 32 + r >= tl.rows_valid) w[r] = 0u;
      }
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) a2 = max_u16x2(a2, w[r] & 0x7FFF7FFFu);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar);  // slot fully read by this warp
    const uint32_t a_lo = a2 & 0xFFFFu;
    const uint32_t a_hi = a2 >> 16;
    const bool nan_lo = a_lo >= 0x7F80u;
    const bool nan_hi = a_hi >= 0x7F80u;
    const int e_lo = nan_lo ? 0 : scale_exponent<FMT>(a_lo, p.rule);
    const int e_hi = nan_hi ? 0 : scale_exponent<FMT>(a_hi, p.rule);
    const float m_lo = pow2_neg(e_lo);
    const float m_hi = pow2_neg(e_hi);
    uint32_t q_lo[8], q_hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // rows 4i..4i+3: .x = column 2cp (scale m_lo), .y = column 2cp + 1 (m_hi)
      const float2 s0 = scale_pair(w[4 * i], m_lo, m_hi);
      const float2 s1 = scale_pair(w[4 * i + 1], m_lo, m_hi);
      const float2 s2 = scale_pair(w[4 * i + 2], m_lo, m_hi);
      const float2 s3 = scale_pair(w[4 * i + 3], m_lo, m_hi);
      constexpr int kPairShift = FMT == 4 ? 8 : 16;  // FP4: a code pair in 8 bits
      if constexpr (SR) {
        // the random integer of column 2cp sits in the low half of the
        // random word, that of column 2cp + 1 in the high half
        const float2 g0 = sr_to_grid2<FMT>(s0, rw[4 * i]);
        const float2 g1 = sr_to_grid2<FMT>(s1, rw[4 * i + 1]);
        const float2 g2 = sr_to_grid2<FMT>(s2, rw[4 * i + 2]);
        const float2 g3 = sr_to_grid2<FMT>(s3, rw[4 * i + 3]);
        q_lo[i] = cvt_pair<FMT>(g0.x, g1.x) | (cvt_pair<FMT>(g2.x, g3.x) << kPairShift);
        q_hi[i] = cvt_pair<FMT>(g0.y, g1.y) | (cvt_pair<FMT>(g2.y, g3.y) << kPairShift);
      } else {
        q_lo[i] = cvt_pair<FMT>(s0.x, s1.x) | (cvt_pair<FMT>(s2.x, s3.x) << kPairShift);
        q_hi[i] = cvt_pair<FMT>(s0.y, s1.y) | (cvt_pair<FMT>(s2.y, s3.y) << kPairShift);
      }
      if (nan_lo) q_lo[i] = F::kNanWord;
      if (nan_hi) q_hi[i] = F::kNanWord;
    }
    stage_col_block<FMT, PACKED>(s_q, 2 * cp, rb, q_lo);
    stage_col_block<FMT, PACKED>(s_q, 2 * cp + 1, rb, q_hi);
    if (ok) {
      s_unit_col[unit_offset(2 * cp, rb)] = nan_lo ? kNanScale : static_cast<uint8_t>(e_lo + 127);
      s_unit_col[unit_offset(2 * cp + 1, rb)] =
          nan_hi ? kNanScale : static_cast<uint8_t>(e_hi + 127);
    }
  }
  group_bar(group);  // scale units and transposed codes complete

  // A 64-column FP32 tile writes its half of each scale unit in place, or
  // the whole unit (the other half zero) when no tile to its right exists.
  const bool whole_unit = kCols == 128 || (half == 0 && tl.c0 + 64 >= p.cols);
  if constexpr (ROW) {
    const int64_t tiles_k = (p.cols + 127) / 128;
    const int64_t unit = tl.scale_rt * tiles_k + tl.c0 / 128;
    if (whole_unit) {
      if (lt < 32)
        reinterpret_cast<uint4*>(p.s_row + unit * 512)[lt] =
            reinterpret_cast<const uint4*>(s_unit_row)[lt];
    } else if (lt < kTile) {
      // the two scales of row lt: bytes 2h, 2h + 1 of its 4-byte group
      const int off = unit_offset(lt, 2 * half);
      *reinterpret_cast<uint16_t*>(p.s_row + unit * 512 + off) =
          *reinterpret_cast<const uint16_t*>(s_unit_row + off);
    }
  }
  if constexpr (COL && PACKED) {
    // Packed transposed codes: output row (c0 + c) holds x rows
    // [x_row0, x_row0 + rows_valid) at bytes [scale_rt * kRowBytes, ...),
    // written in 16-byte (FP4) or 8-byte (FP6) pieces.
    constexpr int kRowBytes = kTile * F::kBits / 8;
    constexpr int kPiece = F::kBits == 4 ? 16 : 8;
    constexpr int kPieces = kRowBytes / kPiece;
    const int64_t ldq_bytes = p.ldq_col * F::kBits / 8;
    const int valid_bytes = static_cast<int>(tl.rows_valid) * F::kBits / 8;
#pragma unroll
    for (int i = 0; i < kCols * kPieces / kGroupThreads; ++i) {
      const int idx = i * kGroupThreads + lt;
      const int c = idx / kPieces;
      const int j = idx - c * kPieces;
      if (tl.c0 + c < p.cols && j * kPiece < valid_bytes) {
        uint8_t* dst = p.q_col + (tl.c0 + c) * ldq_bytes + tl.scale_rt * kRowBytes + j * kPiece;
        if constexpr (kPiece == 16) {
          *reinterpret_cast<uint4*>(dst) =
              *reinterpret_cast<const uint4*>(s_q + c * kColPitch + j * kPiece);
        } else {
          *reinterpret_cast<uint2*>(dst) =
              *reinterpret_cast<const uint2*>(s_q + c * kColPitch + j * kPiece);
        }
      }
    }
  }
  if constexpr (COL) {
    const int64_t tiles_k = (p.ldq_col + 127) / 128;
    const int64_t unit = (tl.c0 / 128) * tiles_k + tl.scale_rt;
    if (whole_unit) {
      if (lt < 32)
        reinterpret_cast<uint4*>(p.s_col + unit * 512)[lt] =
            reinterpret_cast<const uint4*>(s_unit_col)[lt];
    } else if (lt < 32) {
      // unit rows [64h, 64h + 64): bytes [8h, 8h + 8) of each 16-byte line
      const int off = lt * 16 + 8 * half;
      *reinterpret_cast<uint2*>(p.s_col + unit * 512 + off) =
          *reinterpret_cast<const uint2*>(s_unit_col + off);
    }
  }
  if constexpr (COL && !PACKED) {
    // Transposed codes: output row (c0 + c), columns [128 * scale_rt,
    // 128 * scale_rt + 128) (dense: x rows [x_row0, x_row0 + 128); grouped:
    // the tile's place in the group's padded segment).
#pragma unroll
    for (int i = 0; i < kCols * 8 / kGroupThreads; ++i) {
      const int idx = i * kGroupThreads + lt;
      const int c = idx >> 3;
      const int j = idx & 7;
      if (tl.c0 + c < p.cols && (GROUPED || j * 16 < tl.rows_valid)) {
        const uint4 q = *reinterpret_cast<const uint4*>(s_q + c * kColPitch + j * 16);
        *reinterpret_cast<uint4*>(p.q_col + (tl.c0 + c) * p.ldq_col + tl.scale_rt * kTile +
                                  j * 16) = q;
      }
    }
  }
}

// Shared memory: the tile ring, then per consumer group the transposed-code
// buffer (columnwise modes only) and two scale units.  WIDE: the 64 KB
// tiles of the rowwise-only FP32 pass.
template <bool COL, bool SR = false, bool WIDE = false>
struct QSmem {
  // consumer groups (round-robin tiles): three for the rowwise-only rings
  // (bf16: six slots, or three of 64 KB with the random integers; FP32:
  // three 64 KB slots), two otherwise
  static constexpr int kGroups = (!COL && (!SR || !WIDE)) ? 3 : 2;
  static constexpr int kThreads = kGroups * kGroupThreads + 32;  // + one producer warp
  // a slot holds the tile of x, plus its 16-bit random integers with SR
  static constexpr int kXBytes = WIDE ? 2 * kTileBytes : kTileBytes;
  static constexpr int kSlotBytes = kXBytes + (SR ? kTileBytes : 0);
  static constexpr int kStages = WIDE ? (SR ? 2 : 3) : SR ? (COL ? 2 : 3) : (COL ? 4 : 6);
  // Tile i lives in slot i % kStages and is consumed by group i % kGroups.
  // Successive users of a slot (tiles i and i + kStages) must belong to the
  // same group: a group can then never wait on a slot's next phase while
  // the slot's current phase is still outstanding, which a parity wait
  // cannot tell apart from a completed phase.
  static_assert(kStages % kGroups == 0, "ring slots must map to one consumer group");
  static constexpr int kOffRing = 0;
  static constexpr int kOffGroupBuf = kOffRing + kStages * kSlotBytes;
  static constexpr int kGroupBufBytes = (COL ? kTile * kColPitch : 0) + 1024;
  static constexpr int kOffBar = kOffGroupBuf + kGroups * kGroupBufBytes;
  static constexpr int kOffMisc = kOffBar + 2 * kStages * 8;
  static constexpr int kOffGroupInfo = kOffMisc + 16;
  static constexpr int kBytes = kOffGroupInfo + int(sizeof(GroupInfo)) + 1024;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

template <int FMT, bool ROW, bool COL, bool GROUPED, bool SR, bool PACKED, bool F32>
__global__ void __launch_bounds__(QSmem<COL, SR, F32 && !COL>::kThreads, 1)
    quantize_kernel(const __grid_constant__ CUtensorMap tmap_x,
                    const __grid_constant__ CUtensorMap tmap_r, const QuantizeParams p) {
  using QSmem = mx::QSmem<COL, SR, F32 && !COL>;
  constexpr int kStages = QSmem::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + QSmem::kOffBar);
  uint64_t* empty = full + kStages;
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + QSmem::kOffMisc);
  GroupInfo* gi = reinterpret_cast<GroupInfo*>(smem + QSmem::kOffGroupInfo);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int kGroups = QSmem::kGroups;
  constexpr int kProducerWarp = kGroups * kGroupThreads / 32;
  constexpr int kCols = kTileCols<F32, COL>;
  // bytes one tile brings in: x, plus the random integers with SR (2 bytes
  // per column of the tile)
  constexpr uint32_t kTxBytes = QSmem::kXBytes + (SR ? kTile * kCols * 2 : 0);
  // Copies in flight per block, fewer than the ring holds (landed tiles
  // still fill the whole ring): three of six in the dense bf16 rowwise
  // pass, three of four in every pass with columns, two of three in the
  // dense FP32 and stochastic-rounding rowwise passes.  Measured back to
  // back: bf16 rowwise
  // 16384x8192 66.4 us against 73.6 with all six in flight (two 66.1, four
  // 69.5, five 71.6), columnwise 67.6-68.0 against 69.5-69.9, FP32 rowwise
  // 103.8-104.3 against 106.4, grouped columnwise 65536x7168 (64 experts)
  // 221 against 225 us (two: 236); 4096x4096 bf16 rowwise with a clean L2
  // 13.3 against 14.6 us.  The grouped rowwise passes keep the whole ring
  // in flight (bf16: 207 us that way, 219 with three), as do the two-slot
  // rings of stochastic rounding with columns.  The bf16 stochastic-rounding
  // rowwise pass (three 64 KB slots, two copies in flight, three groups)
  // measured 104.3-105.2 us against 108.5-108.8 with two slots and two
  // groups (E5M2, 16384x8192), its whole ring in flight 106.4.
  constexpr int kWindow = kStages <= 2 ? kStages
                          : kStages == 4 ? 3
                          : GROUPED      ? kStages
                          : kStages == 3 ? 2
                                         : 3;

  if (warp == kProducerWarp && lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGroupThreads / 32);  // one arrival per consumer warp
    }
    *s_abort = 0u;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_x);
    if constexpr (SR) tma_prefetch_desc(&tmap_r);
  }
  pdl_wait();  // the input, the offsets and the outputs may belong to the previous kernel
  pdl_launch_dependents();
  if constexpr (GROUPED) group_tile_prefix(p.offsets, p.groups, p.rows, gi->off, gi->tiles, &gi->valid);
  __syncthreads();


  const int64_t col_tiles = (p.cols + kCols - 1) / kCols;
  int64_t num_tiles;
  if constexpr (GROUPED) {
    // columnwise: the padded segments must also fit in the q_col matrix
    const bool fits = !COL || (gi->valid && static_cast<int64_t>(gi->tiles[p.groups]) * kTile <=
                                                 p.ldq_col);
    if (!gi->valid || !fits) {
      if (blockIdx.x == 0 && tid == 0) record_device_status(p.status, MX_DEV_BAD_OFFSETS);
      num_tiles = 0;
    } else {
      num_tiles = static_cast<int64_t>(gi->tiles[p.groups]) * col_tiles;
    }
  } else {
    num_tiles = ((p.rows + kTile - 1) / kTile) * col_tiles;
  }

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int64_t issued = 0;
      int g_hint = 0;
      for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x, ++issued) {
        const uint32_t s = static_cast<uint32_t>(issued % kStages);
        const uint32_t ph = static_cast<uint32_t>((issued / kStages) & 1);
        if (!mbar_wait(&empty[s], ph ^ 1u, s_abort, p.status, p.wait_limit_ns)) break;
        if (kWindow < kStages && issued >= kWindow) {
          // tile issued - kWindow has landed (its slot is not refilled
          // before tile issued - kWindow + kStages, which comes later)
          const int64_t j = issued - kWindow;
          if (!mbar_wait(&full[j % kStages], static_cast<uint32_t>((j / kStages) & 1), s_abort,
                         p.status, p.wait_limit_ns))
            break;
        }
        const Tile tl = tile_of<GROUPED, ROW, COL, kCols>(p, t, col_tiles, gi, g_hint);
        mbar_arrive_expect_tx(&full[s], kTxBytes);
        uint8_t* slot = smem + QSmem::kOffRing + s * QSmem::kSlotBytes;
        const int32_t ry = static_cast<int32_t>(tl.x_row0);
        // boxes of 128 rows x 128 bytes (128-byte swizzle), 16 KB apart: 64
        // bf16 or 32 FP32 columns each; the random integers in boxes of 64
        // columns after x
        constexpr int kBoxCols = F32 ? 32 : 64;
        for (int b = 0; b < kCols / kBoxCols; ++b)
          tma_load_2d(slot + b * (kTileBytes / 2), &tmap_x, &full[s],
                      static_cast<int32_t>(tl.c0) + kBoxCols * b, ry);
        if constexpr (SR) {
          for (int b = 0; b < kCols / 64; ++b)
            tma_load_2d(slot + QSmem::kXBytes + b * (kTileBytes / 2), &tmap_r, &full[s],
                        static_cast<int32_t>(tl.c0) + 64 * b, ry);
        }
      }
      // every issued copy lands before the block exits
      for (int s = 0; s < kStages; ++s) {
        const int64_t fills = issued > s ? (issued - s + kStages - 1) / kStages : 0;
        if (fills)
          mbar_wait(&full[s], static_cast<uint32_t>((fills - 1) & 1), s_abort, p.status,
                    p.wait_limit_ns, true);
      }
    }
  } else {
    const int group = warp / (kGroupThreads / 32);
    const int lt = tid - group * kGroupThreads;
    uint8_t* gbuf = smem + QSmem::kOffGroupBuf + group * QSmem::kGroupBufBytes;
    uint8_t* s_q = gbuf;
    uint8_t* s_unit_row = gbuf + (COL ? kTile * kColPitch : 0);
    uint8_t* s_unit_col = s_unit_row + 512;
    int64_t i = group;  // this block's tile counter; the group takes every kGroups-th tile
    int g_hint = 0;
    for (int64_t t = blockIdx.x + group * static_cast<int64_t>(gridDim.x); t < num_tiles;
         t += kGroups * static_cast<int64_t>(gridDim.x), i += kGroups) {
      const uint32_t s = static_cast<uint32_t>(i % kStages);
      const uint32_t ph = static_cast<uint32_t>((i / kStages) & 1);
      const Tile tl = tile_of<GROUPED, ROW, COL, kCols>(p, t, col_tiles, gi, g_hint);
      group_bar(group);  // the group's previous tile is fully written out
      if (lt < 128) {
        if (ROW) reinterpret_cast<uint32_t*>(s_unit_row)[lt] = 0u;
        if (COL) reinterpret_cast<uint32_t*>(s_unit_col)[lt] = 0u;
      }
      const bool got = mbar_wait(&full[s], ph, s_abort, p.status, p.wait_limit_ns);
      // scale units zeroed; a wait that gave up anywhere stops the whole group
      if (group_bar_any(group, !got)) break;
      const uint8_t* slot = smem + QSmem::kOffRing + s * QSmem::kSlotBytes;
      quantize_tile<FMT, ROW, COL, GROUPED, SR, PACKED, F32>(p, tl, slot, slot + QSmem::kXBytes, s_q,
                                                            s_unit_row, s_unit_col, &empty[s],
                                                            group, lt);
    }
  }
}

// One launch over `tiles` tiles (an upper bound for grouped launches): one
// persistent block per SM, fewer for small inputs.
template <int FMT, bool ROW, bool COL, bool GROUPED, bool SR = false, bool PACKED = false,
          bool F32 = false>
cudaError_t launch_one(const QuantizeParams& p, const CUtensorMap& tmap, const CUtensorMap& tmap_r,
                       int64_t tiles, int num_sms, cudaStream_t stream) {
  auto kern = quantize_kernel<FMT, ROW, COL, GROUPED, SR, PACKED, F32>;
  using QSmem = mx::QSmem<COL, SR, F32 && !COL>;
  static PerDeviceOnce setup;
  const cudaError_t err = setup.run([&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, QSmem::kBytes);
  });
  if (err != cudaSuccess) return err;
  const int64_t grid = tiles < num_sms ? tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(QSmem::kThreads);
  cfg.dynamicSmemBytes = QSmem::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmap, tmap_r, p);
}

template <int FMT, bool PACKED, bool F32>
cudaError_t launch_dense(const QuantizeParams& p, const CUtensorMap& tmap_x,
                         const CUtensorMap* tmap_r, int64_t tiles, int num_sms,
                         cudaStream_t stream) {
  const bool row = p.q_row != nullptr;
  const bool col = p.q_col != nullptr;
  const CUtensorMap& tr = tmap_r ? *tmap_r : tmap_x;
  if (tmap_r) {  // stochastic rounding
    if (row && col)
      return launch_one<FMT, true, true, false, true, PACKED, F32>(p, tmap_x, tr, tiles, num_sms, stream);
    if (row)
      return launch_one<FMT, true, false, false, true, PACKED, F32>(p, tmap_x, tr, tiles, num_sms, stream);
    return launch_one<FMT, false, true, false, true, PACKED, F32>(p, tmap_x, tr, tiles, num_sms, stream);
  }
  if (row && col)
    return launch_one<FMT, true, true, false, false, PACKED, F32>(p, tmap_x, tr, tiles, num_sms, stream);
  if (row)
    return launch_one<FMT, true, false, false, false, PACKED, F32>(p, tmap_x, tr, tiles, num_sms, stream);
  return launch_one<FMT, false, true, false, false, PACKED, F32>(p, tmap_x, tr, tiles, num_sms, stream);
}

// Dense quantization of a bf16 (F32 false) or FP32 input: every element
// format and storage, round to nearest even or (tmap_r given) stochastic
// rounding.
template <bool F32>
cudaError_t launch_quantize_dense(const QuantizeParams& p, const CUtensorMap& tmap_x,
                                  const CUtensorMap* tmap_r, int num_sms, cudaStream_t stream) {
  if (p.rows == 0 || p.cols == 0) return cudaSuccess;
  constexpr int kCols = kTileCols<F32, true>;  // the narrowest tile: an upper bound
  const int64_t tiles = ((p.rows + kTile - 1) / kTile) * ((p.cols + kCols - 1) / kCols);
  switch (p.fmt) {
    case 0: return launch_dense<0, false, F32>(p, tmap_x, tmap_r, tiles, num_sms, stream);
    case 1: return launch_dense<1, false, F32>(p, tmap_x, tmap_r, tiles, num_sms, stream);
    case 2: return launch_dense<2, false, F32>(p, tmap_x, tmap_r, tiles, num_sms, stream);
    case 3: return launch_dense<3, false, F32>(p, tmap_x, tmap_r, tiles, num_sms, stream);
    case 4: return launch_dense<4, false, F32>(p, tmap_x, tmap_r, tiles, num_sms, stream);
    // packed storage of the 6- and 4-bit codes
    case 5: return launch_dense<2, true, F32>(p, tmap_x, tmap_r, tiles, num_sms, stream);
    case 6: return launch_dense<3, true, F32>(p, tmap_x, tmap_r, tiles, num_sms, stream);
    case 7: return launch_dense<4, true, F32>(p, tmap_x, tmap_r, tiles, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Grouped quantization (FP8 codes) of a bf16 or FP32 input.
template <bool F32>
cudaError_t launch_quantize_groups(const QuantizeParams& p, const CUtensorMap& tmap_x,
                                   int num_sms, cudaStream_t stream) {
  if (p.cols == 0) return cudaSuccess;
  if (p.fmt > 1) return cudaErrorNotSupported;  // grouped: FP8 codes
  constexpr int kCols = kTileCols<F32, true>;  // the narrowest tile: an upper bound
  // upper bound of the padded row tiles; the kernel computes the exact count
  const int64_t tiles = ((p.rows + kTile - 1) / kTile + p.groups) * ((p.cols + kCols - 1) / kCols);
  const bool row = p.q_row != nullptr;
  const bool col = p.q_col != nullptr;
  const CUtensorMap& x = tmap_x;
  if (p.fmt == 0) {
    if (row && col) return launch_one<0, true, true, true, false, false, F32>(p, x, x, tiles, num_sms, stream);
    if (row) return launch_one<0, true, false, true, false, false, F32>(p, x, x, tiles, num_sms, stream);
    return launch_one<0, false, true, true, false, false, F32>(p, x, x, tiles, num_sms, stream);
  }
  if (row && col) return launch_one<1, true, true, true, false, false, F32>(p, x, x, tiles, num_sms, stream);
  if (row) return launch_one<1, true, false, true, false, false, F32>(p, x, x, tiles, num_sms, stream);
  return launch_one<1, false, true, true, false, false, F32>(p, x, x, tiles, num_sms, stream);
}

}  // namespace
}  // namespace mx
