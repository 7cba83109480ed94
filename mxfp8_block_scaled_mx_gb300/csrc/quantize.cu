// quantize.cu -- MX quantization kernels (bf16 -> E4M3 / E5M2 codes plus
// E8M0 block scales in the swizzled tensor-core layout).
//
// "Low-Precision GPU Programming" (leetllm.com): section "Microscaling: the
// two-row experiment" (32-element blocks, one E8M0 power-of-two scale per
// block, both orientations from the original wide data) and section
// "Numerical hazards: subnormals, saturation, and rounding" (round to
// nearest even, subnormals kept, saturation after rounding).
//
// One block of 256 threads owns a 128-row x 128-column tile of x.  Each
// thread issues eight coalesced 16-byte loads up front.
//  - Rowwise: the four lanes that hold one 32-element block reduce its amax
//    with two xor-shuffles, derive the scale exponent from the bf16 bit
//    pattern, scale by an exact power of two and convert pairs with the
//    hardware cvt.rn.satfinite instruction.  The tile's 128 x 4 scales form
//    exactly one 512-byte swizzled unit, assembled in shared memory and
//    written with one coalesced store.
//  - Columnwise: the tile is staged in shared memory; each thread reduces
//    and encodes two adjacent columns of a 32-row block (one 32-bit shared
//    load and one SIMD max per row), the codes are transposed in shared
//    memory and written back as 128-byte rows of the [cols, rows] output,
//    again with one 512-byte scale unit per tile.
#include <cuda_runtime.h>

#include <cstdint>

#include "groups.cuh"
#include "kernels.h"
#include "status.cuh"

namespace mx {
namespace {

constexpr int kTile = 128;          // rows and columns of x per block
constexpr int kThreads = 256;
constexpr int kColPitch = 144;      // bytes per transposed code row in smem (conflict-free)

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Per-halfword unsigned max of two packed pairs (one SIMD instruction).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest magnitude bit pattern (sign cleared) among the 8 bf16 of v.  For
// non-NaN bf16 the unsigned order of these patterns is the order of |x|;
// NaN patterns sort above +Inf (0x7F80).
__device__ __forceinline__ uint32_t amax_bits8(const uint4 v) {
  uint32_t m = max_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  m = max_u16x2(m, max_u16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

// Scale exponent e of a block with finite amax (bit pattern `a`):
// floor rule e = floor(log2 amax) - emax_elem; the ceil rule adds one when
// the significand of amax exceeds 1.75 (= max / 2^emax_elem for both E4M3
// and E5M2).  amax = 0 gives e = 0 (S = 1).  Clamped to [-127, 127].
__device__ __forceinline__ int scale_exponent(uint32_t a, int emax, int rule) {
  if (a == 0) return 0;
  const uint32_t ef = a >> 7;
  const uint32_t mant = a & 0x7Fu;
  int fl;
  bool above;
  if (ef != 0) {
    fl = static_cast<int>(ef) - 127;
    above = mant > 0x60u;
  } else {  // bf16 subnormal: value = mant * 2^-133
    const int p = 31 - __clz(mant);
    fl = p - 133;
    above = 4u * mant > (7u << p);
  }
  int e = fl - emax + ((rule == 1 && above) ? 1 : 0);
  return min(max(e, -127), 127);
}

// 2^-e as a float (exact: e in [-127, 127] keeps the exponent normal).
__device__ __forceinline__ float pow2_neg(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// Two floats -> two FP8 codes, RNE with saturation to the finite range;
// `lo` lands in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
  uint16_t r;
  if constexpr (FMT == 0) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

// Two bf16 packed in a word -> two codes (16 bits), after an exact scaling.
template <int FMT>
__device__ __forceinline__ uint32_t encode_word(uint32_t w, float mul) {
  const float lo = __fmul_rn(__uint_as_float(w << 16), mul);
  const float hi = __fmul_rn(__uint_as_float(w & 0xFFFF0000u), mul);
  return cvt_pair<FMT>(lo, hi);
}

template <int FMT>
__device__ __forceinline__ uint2 encode8(const uint4 v, float mul) {
  uint2 r;
  r.x = encode_word<FMT>(v.x, mul) | (encode_word<FMT>(v.y, mul) << 16);
  r.y = encode_word<FMT>(v.z, mul) | (encode_word<FMT>(v.w, mul) << 16);
  return r;
}

constexpr uint32_t kNanCode4 = 0x7F7F7F7Fu;  // four NaN codes
constexpr uint8_t kNanScale = 0xFF;

// Byte offset of (local row r, local block c) inside a 512-byte scale unit.
__device__ __forceinline__ int unit_offset(int r, int c) {
  return (r & 31) * 16 + (r >> 5) * 4 + c;
}

struct TileCoords {
  int64_t x_row0;       // first row of x held by this block
  int64_t rows_valid;   // rows of the tile that exist (<= 128)
  int64_t scale_rt;     // row-tile index of the rowwise scale unit
};

template <int FMT, bool ROW, bool COL>
__device__ __forceinline__ void quantize_tile(const QuantizeParams& p, const TileCoords tc,
                                              int64_t c0, uint8_t* smem) {
  constexpr int emax = FMT == 0 ? 8 : 15;
  const int tid = threadIdx.x;
  uint8_t* s_unit_row = smem;              // 512 B
  uint8_t* s_unit_col = smem + 512;        // 512 B
  uint32_t* s_x = reinterpret_cast<uint32_t*>(smem + 1024);  // 128 rows x 64 bf16 pairs
  uint8_t* s_q = smem + 1024 + kTile * kTile * 2;             // 128 x 144 B

  // Zero the scale units (padding entries stay 0).
  if (tid < 128) {
    if (ROW) reinterpret_cast<uint32_t*>(s_unit_row)[tid] = 0u;
    if (COL) reinterpret_cast<uint32_t*>(s_unit_col)[tid] = 0u;
  }

  // Thread t holds the 8-column chunk t % 16 of rows t / 16 + 16 * it.
  const int ch = tid & 15;
  const int lr0 = tid >> 4;
  const int64_t gc = c0 + ch * 8;
  const bool col_ok = gc < p.cols;
  const uint16_t* xp = p.x + (tc.x_row0 + lr0) * p.ldx + gc;
  const int64_t x_step = 16 * p.ldx;
  uint4 v[8];
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const bool ok = col_ok && lr0 + it * 16 < tc.rows_valid;
    v[it] = ok ? ld_stream(xp + it * x_step) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();  // scale units zeroed

  if constexpr (ROW) {
    uint8_t* qp = p.q_row + (tc.x_row0 + lr0) * p.cols + gc;
    const int64_t q_step = 16 * p.cols;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int lr = lr0 + it * 16;
      const bool ok = col_ok && lr < tc.rows_valid;
      // the four lanes holding one 32-element block share its amax
      uint32_t a = amax_bits8(v[it]);
      a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
      a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
      uint2 codes;
      uint8_t sbyte;
      if (a >= 0x7F80u) {  // NaN or Inf in the block
        codes = make_uint2(kNanCode4, kNanCode4);
        sbyte = kNanScale;
      } else {
        const int e = scale_exponent(a, emax, p.rule);
        codes = encode8<FMT>(v[it], pow2_neg(e));
        sbyte = static_cast<uint8_t>(e + 127);
      }
      if (ok) {
        *reinterpret_cast<uint2*>(qp + it * q_step) = codes;
        if ((tid & 3) == 0) s_unit_row[unit_offset(lr, ch >> 2)] = sbyte;
      }
    }
  }

  if constexpr (COL) {
    // Stage the tile: row lr holds 64 bf16 pairs (256 bytes).
#pragma unroll
    for (int it = 0; it < 8; ++it)
      *reinterpret_cast<uint4*>(s_x + (lr0 + it * 16) * 64 + ch * 4) = v[it];
  }
  __syncthreads();

  if constexpr (COL) {
    // Thread t: columns 2*(t % 64) and 2*(t % 64) + 1, 32-row block t / 64.
    // One 32-bit shared load gives both columns of a row, so the amax of
    // the two column blocks is one SIMD max per row.
    const int cp = tid & 63;
    const int rb = tid >> 6;
    const bool ok = c0 + 2 * cp < p.cols && rb * 32 < tc.rows_valid;
    uint32_t w[32];
    uint32_t a2 = 0;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      w[r] = s_x[(rb * 32 + r) * 64 + cp];
      a2 = max_u16x2(a2, w[r] & 0x7FFF7FFFu);
    }
    const uint32_t a_lo = a2 & 0xFFFFu;
    const uint32_t a_hi = a2 >> 16;
    const bool nan_lo = a_lo >= 0x7F80u;
    const bool nan_hi = a_hi >= 0x7F80u;
    const int e_lo = nan_lo ? 0 : scale_exponent(a_lo, emax, p.rule);
    const int e_hi = nan_hi ? 0 : scale_exponent(a_hi, emax, p.rule);
    const float m_lo = pow2_neg(e_lo);
    const float m_hi = pow2_neg(e_hi);
    uint32_t q_lo[8], q_hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w0 = w[4 * i], w1 = w[4 * i + 1], w2 = w[4 * i + 2], w3 = w[4 * i + 3];
      q_lo[i] = cvt_pair<FMT>(__fmul_rn(__uint_as_float(w0 << 16), m_lo),
                              __fmul_rn(__uint_as_float(w1 << 16), m_lo)) |
                (cvt_pair<FMT>(__fmul_rn(__uint_as_float(w2 << 16), m_lo),
                               __fmul_rn(__uint_as_float(w3 << 16), m_lo))
                 << 16);
      q_hi[i] = cvt_pair<FMT>(__fmul_rn(__uint_as_float(w0 & 0xFFFF0000u), m_hi),
                              __fmul_rn(__uint_as_float(w1 & 0xFFFF0000u), m_hi)) |
                (cvt_pair<FMT>(__fmul_rn(__uint_as_float(w2 & 0xFFFF0000u), m_hi),
                               __fmul_rn(__uint_as_float(w3 & 0xFFFF0000u), m_hi))
                 << 16);
      if (nan_lo) q_lo[i] = kNanCode4;
      if (nan_hi) q_hi[i] = kNanCode4;
    }
    uint4* d0 = reinterpret_cast<uint4*>(s_q + (2 * cp) * kColPitch + rb * 32);
    uint4* d1 = reinterpret_cast<uint4*>(s_q + (2 * cp + 1) * kColPitch + rb * 32);
    d0[0] = make_uint4(q_lo[0], q_lo[1], q_lo[2], q_lo[3]);
    d0[1] = make_uint4(q_lo[4], q_lo[5], q_lo[6], q_lo[7]);
    d1[0] = make_uint4(q_hi[0], q_hi[1], q_hi[2], q_hi[3]);
    d1[1] = make_uint4(q_hi[4], q_hi[5], q_hi[6], q_hi[7]);
    if (ok) {
      s_unit_col[unit_offset(2 * cp, rb)] = nan_lo ? kNanScale : static_cast<uint8_t>(e_lo + 127);
      s_unit_col[unit_offset(2 * cp + 1, rb)] =
          nan_hi ? kNanScale : static_cast<uint8_t>(e_hi + 127);
    }
  }
  __syncthreads();

  if constexpr (ROW) {
    if (tid < 32) {
      const int64_t tiles_k = (p.cols + 127) / 128;
      const int64_t unit = tc.scale_rt * tiles_k + c0 / 128;
      reinterpret_cast<uint4*>(p.s_row + unit * 512)[tid] =
          reinterpret_cast<const uint4*>(s_unit_row)[tid];
    }
  }
  if constexpr (COL) {
    // Transposed codes: output row (c0 + c) holds x rows [x_row0, x_row0 + 128).
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = i * kThreads + tid;
      const int c = idx >> 3;
      const int j = idx & 7;
      if (c0 + c < p.cols && j * 16 < tc.rows_valid) {
        const uint4 q = *reinterpret_cast<const uint4*>(s_q + c * kColPitch + j * 16);
        *reinterpret_cast<uint4*>(p.q_col + (c0 + c) * p.rows + tc.x_row0 + j * 16) = q;
      }
    }
    if (tid < 32) {
      const int64_t tiles_k = (p.rows + 127) / 128;
      const int64_t unit = (c0 / 128) * tiles_k + tc.x_row0 / 128;
      reinterpret_cast<uint4*>(p.s_col + unit * 512)[tid] =
          reinterpret_cast<const uint4*>(s_unit_col)[tid];
    }
  }
}

template <int FMT, bool ROW, bool COL>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const QuantizeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kTile;
  TileCoords tc;
  tc.x_row0 = r0;
  tc.rows_valid = ::min(static_cast<int64_t>(kTile), p.rows - r0);
  tc.scale_rt = blockIdx.x;
  quantize_tile<FMT, ROW, COL>(p, tc, c0, smem);
}

// Rowwise quantization of expert-grouped rows.  blockIdx.x walks the
// padded scale row tiles; tile t belongs to group g with
// s_tiles[g] <= t < s_tiles[g+1] and covers rows o_g + 128 (t - s_tiles[g])
// onward, clipped to the group.
template <int FMT>
__global__ void __launch_bounds__(kThreads) quantize_grouped_kernel(const QuantizeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int32_t s_off[kMaxGroups + 1];
  __shared__ int32_t s_tiles[kMaxGroups + 1];
  __shared__ int32_t s_valid;
  group_tile_prefix(p.offsets, p.groups, p.rows, s_off, s_tiles, &s_valid);
  __syncthreads();
  if (!s_valid) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
      record_device_status(p.status, MX_DEV_BAD_OFFSETS);
    return;
  }
  const int32_t t = blockIdx.x;
  if (t >= s_tiles[p.groups]) return;
  const int g = find_group(s_tiles, p.groups, t);
  TileCoords tc;
  tc.x_row0 = static_cast<int64_t>(s_off[g]) + static_cast<int64_t>(t - s_tiles[g]) * kTile;
  tc.rows_valid = ::min(static_cast<int64_t>(kTile), static_cast<int64_t>(s_off[g + 1]) - tc.x_row0);
  tc.scale_rt = t;
  quantize_tile<FMT, true, false>(p, tc, static_cast<int64_t>(blockIdx.y) * kTile, smem);
}

template <int FMT, bool ROW, bool COL>
cudaError_t launch_dense(const QuantizeParams& p, cudaStream_t stream) {
  auto kern = quantize_kernel<FMT, ROW, COL>;
  const int smem = COL ? 1024 + kTile * kTile * 2 + kTile * kColPitch : 1024;
  if (smem > 48 * 1024) {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
  }
  dim3 grid(static_cast<unsigned>((p.rows + kTile - 1) / kTile),
            static_cast<unsigned>((p.cols + kTile - 1) / kTile));
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const QuantizeParams& p, cudaStream_t stream) {
  if (p.rows == 0 || p.cols == 0) return cudaSuccess;
  const bool row = p.q_row != nullptr;
  const bool col = p.q_col != nullptr;
  if (p.fmt == 0) {
    if (row && col) return launch_dense<0, true, true>(p, stream);
    if (row) return launch_dense<0, true, false>(p, stream);
    return launch_dense<0, false, true>(p, stream);
  }
  if (row && col) return launch_dense<1, true, true>(p, stream);
  if (row) return launch_dense<1, true, false>(p, stream);
  return launch_dense<1, false, true>(p, stream);
}

cudaError_t launch_quantize_grouped(const QuantizeParams& p, cudaStream_t stream) {
  if (p.cols == 0) return cudaSuccess;
  const int64_t max_tiles = (p.rows + kTile - 1) / kTile + p.groups;
  dim3 grid(static_cast<unsigned>(max_tiles), static_cast<unsigned>((p.cols + kTile - 1) / kTile));
  if (p.fmt == 0) {
    quantize_grouped_kernel<0><<<grid, kThreads, 1024, stream>>>(p);
  } else {
    quantize_grouped_kernel<1><<<grid, kThreads, 1024, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace mx
