// kernels.h -- launch interface between the C-ABI layer (mx_api.cu) and the
// CUDA kernels (quantize.cu and quantize_f32.cu, which instantiate
// quantize_kernel.cuh; gemm_pair.cu; status.cu).  Not part of the public
// ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace mx {

// Launch attribute of every kernel of the library: programmatic stream
// serialization (the kernels wait for their predecessor with griddepcontrol
// before touching global memory).
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// One-time set-up of a kernel per device (its dynamic shared-memory limit):
// `fn` runs until it first succeeds on the current device.  The flags are
// guarded by a mutex, so concurrent first calls from several host threads
// are safe.
class PerDeviceOnce {
 public:
  template <typename Fn>
  cudaError_t run(Fn&& fn) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDev) return fn();
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev]) return cudaSuccess;
    err = fn();
    if (err == cudaSuccess) done_[dev] = true;
    return err;
  }

 private:
  static constexpr int kMaxDev = 64;
  std::mutex mu_;
  bool done_[kMaxDev] = {};
};

struct QuantizeParams {
  const void* x;       // bf16 or FP32 elements, [rows, cols], leading dimension ldx
                       // (the kernels read x through its tensor map)
  int64_t rows;
  int64_t cols;
  int64_t ldx;
  uint8_t* q_row;      // [rows, cols] codes or nullptr
  uint8_t* s_row;      // swizzled scales of the [rows, cols] operand
  uint8_t* q_col;      // [cols, rows] codes or nullptr
  uint8_t* s_col;      // swizzled scales of the [cols, rows] operand
  int32_t fmt;         // element format: 0 E4M3, 1 E5M2, 2 E2M3, 3 E3M2, 4 E2M1; 5-7 the
                       // last three in packed storage
  int32_t rule;        // 0 = floor, 1 = ceil
  const int32_t* offsets;  // grouped only: device int32[groups + 1]
  int32_t groups;
  uint32_t* status;    // device status word
  uint64_t wait_limit_ns;
  int64_t ldq_col;     // columns of the q_col matrix (dense: rows; grouped: the
                       // 128-padded token capacity, a multiple of 128)
};

// tmap_x: 2-D bf16 tensor map over x (box 64 columns x 128 rows, 128-byte
// swizzle); tmap_r: the same over the 16-bit random integers for stochastic
// rounding, or nullptr for round-to-nearest-even.
cudaError_t launch_quantize(const QuantizeParams& p, const CUtensorMap& tmap_x,
                            const CUtensorMap* tmap_r, int num_sms, cudaStream_t stream);
// Grouped: rowwise (q_row) and/or columnwise (q_col, per-group padded
// segments of 128 columns) quantization of token groups.
cudaError_t launch_quantize_grouped(const QuantizeParams& p, const CUtensorMap& tmap_x,
                                    int num_sms, cudaStream_t stream);
// The same for FP32 x: tmap_x is a 2-D FP32 tensor map (box 32 columns x 128
// rows, 128-byte swizzle); tmap_r as above.
cudaError_t launch_quantize_f32(const QuantizeParams& p, const CUtensorMap& tmap_x,
                                const CUtensorMap* tmap_r, int num_sms, cudaStream_t stream);
cudaError_t launch_quantize_grouped_f32(const QuantizeParams& p, const CUtensorMap& tmap_x,
                                        int num_sms, cudaStream_t stream);

// GEMM modes: dense; grouped by rows of A (each expert owns a range of A
// rows and its own B); grouped along K (each expert owns a 128-aligned
// range of the K columns of A and B and its own output matrix).
constexpr int kModeDense = 0;
constexpr int kModeGroupM = 1;
constexpr int kModeGroupK = 2;

struct GemmParams {
  int64_t m;           // rows of A and Y (grouped by rows: total rows; grouped
                       // along K: rows of A and of each output matrix)
  int64_t n;           // rows of each B (columns of Y)
  int64_t k;           // contraction length, a multiple of 16 (a final block of
                       // 16 is zero-filled past K; grouped along K: unused,
                       // each group's length comes from the offsets)
  int64_t lda;         // columns of the A code matrix (K-contiguous)
  int64_t ldb;         // columns of the B code matrix
  int32_t b_concat;    // grouped by rows: 1 = B is one [n, ldb] matrix with
                       // expert g's operand in columns [g*k, (g+1)*k)
  const uint8_t* sa;   // swizzled scales of A (grouped: per-group padded)
  const uint8_t* sb;   // swizzled scales of B (grouped: one matrix per group)
  void* y;
  int64_t ldy;         // elements
  int32_t y_fp32;      // 1: FP32 output, 0: BF16 output
  int32_t fa;          // tensor-core operand type code (E4M3 0, E5M2 1, E2M3 3, E3M2 4, E2M1 5)
  int32_t fb;
  const int32_t* offsets;  // grouped only: device int32[groups + 1]
  int32_t groups;          // 0 for the dense GEMM
  int32_t mode;            // kModeDense, kModeGroupM or kModeGroupK
  uint32_t* status;
  uint64_t wait_limit_ns;
  int32_t band_m;          // m-tiles per raster band (dense), a multiple of 2
  const float* bias;       // fused epilogue: FP32 bias per output column, or nullptr
  int32_t act;             // fused epilogue: 0 none, 1 SiLU
  int32_t a_bits;          // bits of global storage per A / B code: 8, or 4 / 6 when
  int32_t b_bits;          // packed (the tensor copy counts the global bytes it reads)
};

// Block-pair GEMM (cta_group::2, 256 x 256 pair tiles), all three modes.
// tmap_a / tmap_b: codes, box 128 rows; tmap_sa / tmap_sb: the swizzled
// scale buffers viewed as uint32 [row_tiles][k_tiles][128], boxes of one
// (A) and two (B) 512-byte units.
cudaError_t launch_gemm_pair(const GemmParams& p, const CUtensorMap& tmap_a,
                             const CUtensorMap& tmap_b, const CUtensorMap& tmap_sa,
                             const CUtensorMap& tmap_sb, int num_sms, cudaStream_t stream);

// Clears the bits `bits` of the device status word (atomically, so bits
// set meanwhile by kernels on other streams survive).
cudaError_t launch_status_clear(uint32_t* status, uint32_t bits, cudaStream_t stream);

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace mx
