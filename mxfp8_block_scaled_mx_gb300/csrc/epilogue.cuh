// epilogue.cuh -- the GEMM epilogue of one accumulator share (32 rows x
// BN/2 columns held by one warp): tcgen05.ld of the FP32 accumulator into
// registers, release of the accumulator (callback), optional fused bias and
// SiLU in FP32, conversion to FP32/BF16 (RNE), staging through 2 KB of
// shared memory and coalesced 64-byte row segments to global memory, masked
// at the matrix edge.
#pragma once

#include <cstdint>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace mx {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// t_row: tensor-memory address of this warp's lane quarter and first
// column; grow0/gcol0: output coordinates of that lane 0 / column 0; rows
// >= m_end and columns >= p.n are not stored.  `release` runs once the
// accumulator share is in registers (it must fence and arrive).  `zero`:
// the tile had no K blocks (an expert without tokens), so the output is
// zero and tensor memory is not read.
template <int BN, bool FUSED, typename Release>
__device__ __forceinline__ void epilogue_share(const GemmParams& p, uint32_t t_row,
                                               int64_t grow0, int64_t gcol0, int64_t m_end,
                                               uint8_t* stage_buf, uint32_t lane, bool zero,
                                               Release&& release) {
  constexpr int kCols = BN / 2;
  const int64_t m_end_ = m_end;
  // staged rows are 64 bytes: 16-byte chunk j of row r sits at chunk
  // j ^ ((r >> 1) & 3), which keeps both the row-wise writes and the
  // 4-lanes-per-row reads free of bank conflicts.
  auto chunk_at = [](int r, int j) { return r * 64 + ((j ^ ((r >> 1) & 3)) * 16); };
  // Fused epilogue on local columns [c0, c0 + CNT): z = acc + bias[col]
  // in FP32, then the activation, before the one rounding to the output
  // type.  Every lane reads the same bias address (a broadcast).
  auto fuse = [&](uint32_t* vals, int c0, auto cnt_tag) {
    constexpr int CNT = decltype(cnt_tag)::value;
#pragma unroll
    for (int c4 = 0; c4 < CNT / 4; ++c4) {
      float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
      const int64_t col = gcol0 + c0 + c4 * 4;
      if (p.bias != nullptr && col < p.n) bv = *reinterpret_cast<const float4*>(p.bias + col);
      const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float z = __fadd_rn(__uint_as_float(vals[c4 * 4 + e]), bb[e]);
        if (p.act == 1) {
          // FP32 outputs use the accurate exponential and division; BF16
          // outputs (8 significant bits) the fast exponential and the fast
          // division (approximate reciprocal times z), whose ~1e-6
          // relative error is far below one BF16 ulp.  exp overflow gives
          // z / inf = -0 for very negative z (both forms).
          z = p.y_fp32 ? __fdiv_rn(z, __fadd_rn(1.0f, expf(-z)))
                       : __fdividef(z, __fadd_rn(1.0f, __expf(-z)));
        }
        vals[c4 * 4 + e] = __float_as_uint(z);
      }
    }
  };
  if (p.y_fp32 || FUSED) {
    // Whole share as FP32 in registers; the accumulator is released
    // before any epilogue arithmetic.
    uint32_t v[kCols];
    if (!zero) {
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c)
        tmem_ld_32x32b_x32(t_row + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int c = 0; c < kCols; ++c) v[c] = 0u;
    }
    release();
    if (p.y_fp32) {
      float* y = static_cast<float*>(p.y);
#pragma unroll
      for (int pass = 0; pass < kCols / 16; ++pass) {  // 16 FP32 columns = 64 bytes per row
        if constexpr (FUSED) fuse(&v[pass * 16], pass * 16, std::integral_constant<int, 16>{});
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(stage_buf + chunk_at(lane, j)) =
              make_uint4(v[pass * 16 + 4 * j], v[pass * 16 + 4 * j + 1],
                         v[pass * 16 + 4 * j + 2], v[pass * 16 + 4 * j + 3]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int rr = it * 8 + (lane >> 2);
          const int j = lane & 3;
          const int64_t grow = grow0 + rr;
          const int64_t gcol = gcol0 + pass * 16 + j * 4;
          if (grow < m_end_ && gcol < p.n)
            *reinterpret_cast<uint4*>(y + grow * p.ldy + gcol) =
                *reinterpret_cast<const uint4*>(stage_buf + chunk_at(rr, j));
        }
        __syncwarp();
      }
    } else {
      uint16_t* y = static_cast<uint16_t*>(p.y);
#pragma unroll
      for (int pass = 0; pass < kCols / 32; ++pass) {  // 32 BF16 columns = 64 bytes per row
        if constexpr (FUSED) fuse(&v[pass * 32], pass * 32, std::integral_constant<int, 32>{});
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(v[pass * 32 + 2 * i]),
                             __uint_as_float(v[pass * 32 + 2 * i + 1]));
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(stage_buf + chunk_at(lane, j)) =
              make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int rr = it * 8 + (lane >> 2);
          const int j = lane & 3;
          const int64_t grow = grow0 + rr;
          const int64_t gcol = gcol0 + pass * 32 + j * 8;
          if (grow < m_end_ && gcol < p.n)
            *reinterpret_cast<uint4*>(y + grow * p.ldy + gcol) =
                *reinterpret_cast<const uint4*>(stage_buf + chunk_at(rr, j));
        }
        __syncwarp();
      }
    }
  } else {
    uint32_t w[kCols / 2];
    if (!zero) {
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[c * 16 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
      }
    } else {
#pragma unroll
      for (int i = 0; i < kCols / 2; ++i) w[i] = 0u;
    }
    release();
    uint16_t* y = static_cast<uint16_t*>(p.y);
#pragma unroll
    for (int pass = 0; pass < kCols / 32; ++pass) {  // 32 BF16 columns = 64 bytes per row
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(stage_buf + chunk_at(lane, j)) =
            make_uint4(w[pass * 16 + 4 * j], w[pass * 16 + 4 * j + 1],
                       w[pass * 16 + 4 * j + 2], w[pass * 16 + 4 * j + 3]);
      __syncwarp();
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int rr = it * 8 + (lane >> 2);
        const int j = lane & 3;
        const int64_t grow = grow0 + rr;
        const int64_t gcol = gcol0 + pass * 32 + j * 8;
        if (grow < m_end_ && gcol < p.n)
          *reinterpret_cast<uint4*>(y + grow * p.ldy + gcol) =
              *reinterpret_cast<const uint4*>(stage_buf + chunk_at(rr, j));
      }
      __syncwarp();
    }
  }
}

}  // namespace mx
