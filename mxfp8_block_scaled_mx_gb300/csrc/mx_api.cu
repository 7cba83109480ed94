// mx_api.cu -- the C ABI (include/mx.h): argument validation, TMA tensor
// map encoding through the driver entry point, device status word, and
// kernel launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "kernels.h"
#include "mx.h"

namespace {

// The device status word (one per device, in this module's device memory).
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

struct DeviceState {
  bool ready = false;
  int device = 0;
  int num_sms = 0;
  uint32_t* status = nullptr;  // device address of g_status_word on this device
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
// Dense GEMMs walk their output tiles in bands of this many 128-row tiles
// (n-tiles outer inside a band), so a band of A stays in L2 while B streams.
constexpr int32_t kBandM = 32;

mx_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MX_ERR_CUDA;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return MX_ERR_CUDA;
    st.status = static_cast<uint32_t*>(addr);
    if (cudaMemset(st.status, 0, sizeof(uint32_t)) != cudaSuccess) return MX_ERR_CUDA;
    st.device = dev;
    st.ready = true;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return MX_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = &st;
  return MX_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every non-null pointer of the list points into device memory of device
// `dev` (memory of cudaMalloc or a memory pool on that device).  Host memory
// (pinned, mapped or unregistered), managed memory and the memory of other
// devices -- all reachable through unified addressing -- are refused, so
// the kernels and their tensor copies only ever read this GPU's own memory.
bool all_on_device(int dev, std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (p == nullptr) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      (void)cudaGetLastError();  // clear the (non-sticky) error of the query
      return false;
    }
    if (a.type != cudaMemoryTypeDevice || a.device != dev) return false;
  }
  return true;
}

bool valid_fmt(mx_fmt f) { return f == MX_E4M3 || f == MX_E5M2; }

// GEMM operand formats: FP8 and the MXFP6 / MXFP4 element formats, the
// latter in container or packed storage.
bool valid_gemm_fmt(mx_fmt f) { return f >= MX_E4M3 && f <= MX_E2M1_PACKED; }

bool is_packed(mx_fmt f) { return f >= MX_E2M3_PACKED; }

// Code width in bits.
int code_bits(mx_fmt f) {
  switch (f) {
    case MX_E2M3: case MX_E3M2: case MX_E2M3_PACKED: case MX_E3M2_PACKED: return 6;
    case MX_E2M1: case MX_E2M1_PACKED: return 4;
    default: return 8;
  }
}

// Operand type code of tcgen05.mma.kind::mxf8f6f4 (instruction descriptor
// bits 7-9 / 10-12): E4M3 0, E5M2 1, E2M3 3, E3M2 4, E2M1 5 (either storage).
int32_t mma_type_code(mx_fmt f) {
  switch (f) {
    case MX_E5M2: return 1;
    case MX_E2M3: case MX_E2M3_PACKED: return 3;
    case MX_E3M2: case MX_E3M2_PACKED: return 4;
    case MX_E2M1: case MX_E2M1_PACKED: return 5;
    default: return 0;
  }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// 2-D uint8 tensor map over a [rows, inner] row-major matrix with row stride
// `stride` bytes, tile box {128 bytes, box_rows}, 128-byte swizzle, zero
// fill outside the matrix.
mx_status encode_codes_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows,
                           int64_t stride, uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride)};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// 2-D bf16 tensor map over x[rows, cols] (leading dimension ldx elements),
// box 64 columns x 128 rows (128-byte rows, two boxes per 128 x 128 tile),
// 128-byte swizzle, zero fill outside the matrix.
mx_status encode_bf16_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                          int64_t ldx) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx * 2)};
  cuuint32_t box[2] = {64u, 128u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// 2-D tensor map over an FP32 [rows, cols] matrix with leading dimension
// ldx: box 32 columns x 128 rows (128-byte rows, two boxes per 128 x 64
// tile), 128-byte swizzle, zero fill outside the matrix.
mx_status encode_f32_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                         int64_t ldx) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx * 4)};
  cuuint32_t box[2] = {32u, 128u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// 2-D tensor map over packed 6- or 4-bit codes [rows, inner elements] with
// row stride `stride` bytes, read with the unpacking element type: each run
// of 16 codes lands in 16 bytes of shared memory (the container layout the
// MMA reads), so the shared-memory tile equals that of a container-layout
// operand.  Box {128 elements, box_rows}, 128-byte swizzle, zero fill.
mx_status encode_packed_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows,
                            int64_t stride, uint32_t box_rows, int bits) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride)};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  const CUtensorMapDataType type =
      bits == 4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B;
  CUresult r = g_encode(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// Tensor map of a GEMM code operand [rows, ld elements] in its storage.
mx_status encode_operand_map(CUtensorMap* map, const void* base, mx_fmt f, int64_t ld,
                             int64_t rows) {
  if (is_packed(f))
    return encode_packed_map(map, base, ld, rows, ld * code_bits(f) / 8, 128, code_bits(f));
  return encode_codes_map(map, base, ld, rows, ld, 128);
}

// The swizzled scale buffer of a [rows, k] operand viewed as uint32
// [ceil(rows/128)][ceil(k/128)][128] (one 512-byte unit per 128-row x
// 128-K tile); box of `units` consecutive row tiles at one K tile.
mx_status encode_scale_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k,
                           uint32_t units) {
  const int64_t row_tiles = ceil_div(rows, 128);
  const int64_t k_tiles = ceil_div(k, 128);
  cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(k_tiles),
                        static_cast<cuuint64_t>(row_tiles)};
  cuuint64_t strides[2] = {512u, static_cast<cuuint64_t>(512 * k_tiles)};
  cuuint32_t box[3] = {128u, 1u, units};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// Operand geometry of one GEMM launch: A codes [m, lda] (grouped along K:
// [m, lda] shared by all groups), B codes [b_rows, ldb]; scales swizzled
// over the same shapes.
struct GemmShape {
  int64_t m, n, k;
  int64_t lda, ldb, b_rows;
  int32_t groups = 0;
  const int32_t* d_offsets = nullptr;
  int32_t mode = mx::kModeDense;
  int32_t b_concat = 0;
};

mx_status gemm_common(const GemmShape& g, const uint8_t* a, const uint8_t* sa, mx_fmt fa,
                      const uint8_t* b, const uint8_t* sb, mx_fmt fb, void* y, mx_dtype y_dtype,
                      int64_t ldy, cudaStream_t stream, const float* bias = nullptr,
                      int32_t act = 0) {
  const int64_t m = g.m, n = g.n, k = g.k;
  if (!a || !sa || !b || !sb || !y) return MX_ERR_INVALID_ARG;
  if (m < 0 || n <= 0 || k < 0 || n % 8 != 0 || ldy < n) return MX_ERR_INVALID_ARG;
  // grouped along K, k is the token total that the offsets split; else
  // whole 16-element runs (a final partial block of 16 is zero-padded)
  if (g.mode != mx::kModeGroupK && (k < 16 || k % 16 != 0)) return MX_ERR_INVALID_ARG;
  if (!valid_gemm_fmt(fa) || !valid_gemm_fmt(fb)) return MX_ERR_INVALID_ARG;
  if (y_dtype != MX_BF16 && y_dtype != MX_FP32) return MX_ERR_INVALID_ARG;
  if (m > INT32_MAX || g.b_rows > INT32_MAX || k > INT32_MAX || g.lda > INT32_MAX ||
      g.ldb > INT32_MAX)
    return MX_ERR_UNSUPPORTED;
  // the kernels index their 256x256 work units in 32 bits
  {
    const int64_t m_tiles = ceil_div(m, 128);
    int64_t units = g.mode == mx::kModeGroupM ? (m_tiles + g.groups + 1) / 2 + g.groups
                                              : (m_tiles + 1) / 2;
    units *= ceil_div(n, 256);
    if (g.mode == mx::kModeGroupK) units *= g.groups;
    if (units > INT32_MAX) return MX_ERR_UNSUPPORTED;
  }
  const int64_t elt = y_dtype == MX_FP32 ? 4 : 2;
  if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(y) ||
      (ldy * elt) % 16 != 0 || g.lda % 16 != 0 || g.ldb % 16 != 0)
    return MX_ERR_MISALIGNED;
  // packed operands: whole 128-element K tiles (the unpacking tensor copy
  // reads rows of a multiple of 128 elements) and 32-byte aligned rows
  if ((is_packed(fa) && (g.lda % 128 != 0 || (g.mode != mx::kModeGroupK && k % 128 != 0))) ||
      (is_packed(fb) && (g.ldb % 128 != 0 || (g.mode != mx::kModeGroupK && k % 128 != 0))))
    return MX_ERR_INVALID_ARG;
  if ((is_packed(fa) && (reinterpret_cast<uintptr_t>(a) & 31u) != 0) ||
      (is_packed(fb) && (reinterpret_cast<uintptr_t>(b) & 31u) != 0))
    return MX_ERR_MISALIGNED;
  DeviceState* st = nullptr;
  mx_status s = device_state(&st);
  if (s != MX_OK) return s;
  if (m == 0) return MX_OK;
  if (!all_on_device(st->device, {a, sa, b, sb, y, bias, g.d_offsets})) return MX_ERR_INVALID_ARG;

  mx::GemmParams p{};
  p.m = m;
  p.n = n;
  p.k = k;
  p.lda = g.lda;
  p.ldb = g.ldb;
  p.b_concat = g.b_concat;
  p.sa = sa;
  p.sb = sb;
  p.y = y;
  p.ldy = ldy;
  p.y_fp32 = y_dtype == MX_FP32 ? 1 : 0;
  p.fa = mma_type_code(fa);
  p.fb = mma_type_code(fb);
  p.offsets = g.d_offsets;
  p.groups = g.groups;
  p.mode = g.mode;
  p.status = st->status;
  p.wait_limit_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.bias = bias;
  p.act = act;
  p.band_m = kBandM;
  p.a_bits = is_packed(fa) ? code_bits(fa) : 8;
  p.b_bits = is_packed(fb) ? code_bits(fb) : 8;

  // Block pairs (cta_group::2, 256x256 pair tiles): each block loads 128
  // rows of A and 128 of the 256 rows of the B tile; the scale buffers are
  // viewed as grids of 512-byte units, A's with the per-group padded row
  // bound when grouped by rows.
  CUtensorMap ta, tb, tsa, tsb;
  const int64_t a_scale_rows = g.mode == mx::kModeGroupM ? (ceil_div(m, 128) + g.groups) * 128 : m;
  if ((s = encode_operand_map(&ta, a, fa, g.lda, m)) != MX_OK) return s;
  if ((s = encode_operand_map(&tb, b, fb, g.ldb, g.b_rows)) != MX_OK) return s;
  if ((s = encode_scale_map(&tsa, sa, a_scale_rows, g.lda, 1)) != MX_OK) return s;
  if ((s = encode_scale_map(&tsb, sb, g.b_rows, g.ldb, 2)) != MX_OK) return s;
  const cudaError_t err = mx::launch_gemm_pair(p, ta, tb, tsa, tsb, st->num_sms, stream);
  if (err == cudaErrorNotSupported) return MX_ERR_UNSUPPORTED;
  return err == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

GemmShape dense_shape(int64_t m, int64_t n, int64_t k) {
  GemmShape g;
  g.m = m;
  g.n = n;
  g.k = k;
  g.lda = k;
  g.ldb = k;
  g.b_rows = n;
  return g;
}

}  // namespace

extern "C" {

size_t mx_scale_bytes(int64_t rows, int64_t k) {
  if (rows < 0 || k < 0 || k % 16 != 0) return 0;
  return static_cast<size_t>(ceil_div(rows, 128) * 128 * ceil_div(ceil_div(k, 32), 4) * 4);
}

size_t mx_grouped_scale_bytes(int64_t total_rows, int32_t groups, int64_t k) {
  if (total_rows < 0 || groups < 0 || k < 0 || k % 16 != 0) return 0;
  return static_cast<size_t>((ceil_div(total_rows, 128) + groups) * 128 * ceil_div(k, 128) * 4);
}

}  // extern "C"

namespace {

mx_status quantize_common(const void* x, mx_dtype x_dtype, int64_t rows, int64_t cols,
                          int64_t ldx, const uint16_t* rbits, int64_t ldr, mx_fmt fmt,
                          mx_axis axis, mx_scale_rule rule, uint8_t* q_row, uint8_t* s_row,
                          uint8_t* q_col, uint8_t* s_col, cudaStream_t stream) {
  if (x_dtype != MX_BF16 && x_dtype != MX_FP32) return MX_ERR_INVALID_ARG;
  const bool f32 = x_dtype == MX_FP32;
  if (!valid_gemm_fmt(fmt) || (rule != MX_SCALE_FLOOR && rule != MX_SCALE_CEIL))
    return MX_ERR_INVALID_ARG;
  if (axis != MX_ROWWISE && axis != MX_COLWISE && axis != MX_BOTH) return MX_ERR_INVALID_ARG;
  const bool row = axis & MX_ROWWISE;
  const bool col = axis & MX_COLWISE;
  if (!x || (row && (!q_row || !s_row)) || (col && (!q_col || !s_col))) return MX_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ldx < cols || cols % 8 != 0) return MX_ERR_INVALID_ARG;
  if (rbits && ldr < cols) return MX_ERR_INVALID_ARG;
  // the blocked axis: whole 16-element runs (16-byte code rows; a final
  // partial block of 16 is zero-padded), whole blocks in packed storage
  const int64_t k_unit = is_packed(fmt) ? 32 : 16;
  if (row && cols % k_unit != 0) return MX_ERR_INVALID_ARG;
  if (col && rows % k_unit != 0) return MX_ERR_INVALID_ARG;
  if (ceil_div(cols, 128) > 65535) return MX_ERR_UNSUPPORTED;
  // the kernels number their tiles (128 rows x 128 bf16 or 64 FP32 columns) in 32 bits
  const int64_t col_tiles = ceil_div(cols, f32 ? 64 : 128);
  if (cols > 0 && ceil_div(rows, 128) > static_cast<int64_t>(UINT32_MAX) / col_tiles)
    return MX_ERR_UNSUPPORTED;
  // rows of x start on 16-byte boundaries
  if (!aligned16(x) || ldx % (f32 ? 4 : 8) != 0) return MX_ERR_MISALIGNED;
  if (rbits && (!aligned16(rbits) || ldr % 8 != 0)) return MX_ERR_MISALIGNED;
  if ((row && (!aligned16(q_row) || !aligned16(s_row))) ||
      (col && (!aligned16(q_col) || !aligned16(s_col))))
    return MX_ERR_MISALIGNED;
  DeviceState* st = nullptr;
  mx_status s = device_state(&st);
  if (s != MX_OK) return s;
  mx::QuantizeParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.ldx = ldx;
  p.q_row = row ? q_row : nullptr;
  p.s_row = row ? s_row : nullptr;
  p.q_col = col ? q_col : nullptr;
  p.s_col = col ? s_col : nullptr;
  p.fmt = fmt;
  p.rule = rule;
  p.status = st->status;
  p.wait_limit_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.ldq_col = rows;
  if (rows == 0 || cols == 0) return MX_OK;
  if (!all_on_device(st->device, {x, rbits, p.q_row, p.s_row, p.q_col, p.s_col}))
    return MX_ERR_INVALID_ARG;
  CUtensorMap tmap, tmap_r;
  s = f32 ? encode_f32_map(&tmap, x, cols, rows, ldx) : encode_bf16_map(&tmap, x, cols, rows, ldx);
  if (s != MX_OK) return s;
  // the random integers are 16-bit like bf16: the bf16 box geometry
  if (rbits && (s = encode_bf16_map(&tmap_r, rbits, cols, rows, ldr)) != MX_OK) return s;
  const CUtensorMap* tr = rbits ? &tmap_r : nullptr;
  const cudaError_t err = f32 ? mx::launch_quantize_f32(p, tmap, tr, st->num_sms, stream)
                              : mx::launch_quantize(p, tmap, tr, st->num_sms, stream);
  return err == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace

extern "C" {

mx_status mx_quantize(const void* x, mx_dtype x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                      mx_fmt fmt, mx_axis axis, mx_scale_rule rule, uint8_t* q_row,
                      uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, cudaStream_t stream) {
  return quantize_common(x, x_dtype, rows, cols, ldx, nullptr, 0, fmt, axis, rule, q_row, s_row,
                         q_col, s_col, stream);
}

mx_status mx_quantize_sr(const void* x, mx_dtype x_dtype, int64_t rows, int64_t cols, int64_t ldx,
                         const uint16_t* rbits, int64_t ldr, mx_fmt fmt, mx_axis axis,
                         mx_scale_rule rule, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                         uint8_t* s_col, cudaStream_t stream) {
  if (!rbits) return MX_ERR_INVALID_ARG;
  return quantize_common(x, x_dtype, rows, cols, ldx, rbits, ldr, fmt, axis, rule, q_row, s_row,
                         q_col, s_col, stream);
}

mx_status mx_quantize_grouped(const void* x, mx_dtype x_dtype, int64_t total_rows, int64_t cols,
                              int64_t ldx, mx_fmt fmt, mx_scale_rule rule, int32_t groups,
                              const int32_t* d_offsets, uint8_t* q, uint8_t* s,
                              cudaStream_t stream) {
  if (!q || !s) return MX_ERR_INVALID_ARG;
  return mx_quantize_grouped_ex(x, x_dtype, total_rows, cols, ldx, fmt, MX_ROWWISE, rule, groups,
                                d_offsets, q, s, nullptr, 0, nullptr, stream);
}

int64_t mx_grouped_cols_capacity(int64_t total_rows, int32_t groups) {
  if (total_rows < 0 || groups < 0) return 0;
  return (total_rows / 128 + groups) * 128;
}

mx_status mx_quantize_grouped_ex(const void* x, mx_dtype x_dtype, int64_t total_rows,
                                 int64_t cols, int64_t ldx, mx_fmt fmt, mx_axis axis,
                                 mx_scale_rule rule, int32_t groups, const int32_t* d_offsets,
                                 uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, int64_t ldq_col,
                                 uint8_t* s_col, cudaStream_t stream) {
  if (x_dtype != MX_BF16 && x_dtype != MX_FP32) return MX_ERR_INVALID_ARG;
  const bool f32 = x_dtype == MX_FP32;
  if (!valid_gemm_fmt(fmt) || (rule != MX_SCALE_FLOOR && rule != MX_SCALE_CEIL))
    return MX_ERR_INVALID_ARG;
  if (!valid_fmt(fmt)) return MX_ERR_UNSUPPORTED;  // grouped: FP8 codes
  if (axis != MX_ROWWISE && axis != MX_COLWISE && axis != MX_BOTH) return MX_ERR_INVALID_ARG;
  const bool row = axis & MX_ROWWISE;
  const bool col = axis & MX_COLWISE;
  if (!x || !d_offsets || (row && (!q_row || !s_row)) || (col && (!q_col || !s_col)))
    return MX_ERR_INVALID_ARG;
  if (groups < 1 || groups > 1000) return MX_ERR_INVALID_ARG;
  if (total_rows < 0 || total_rows > INT32_MAX || cols < 0 || ldx < cols || cols % 8 != 0)
    return MX_ERR_INVALID_ARG;
  if (row && cols % 16 != 0) return MX_ERR_INVALID_ARG;
  if (col && (ldq_col <= 0 || ldq_col % 128 != 0)) return MX_ERR_INVALID_ARG;
  if (ceil_div(cols, 128) > 65535) return MX_ERR_UNSUPPORTED;
  // the columnwise pass numbers its tiles (128 rows x 128 bf16 or 64 FP32
  // columns) in 32 bits
  if (col && (ceil_div(total_rows, 128) + groups) * ceil_div(cols, f32 ? 64 : 128) > UINT32_MAX)
    return MX_ERR_UNSUPPORTED;
  if (!aligned16(x) || ldx % (f32 ? 4 : 8) != 0) return MX_ERR_MISALIGNED;
  if ((row && (!aligned16(q_row) || !aligned16(s_row))) ||
      (col && (!aligned16(q_col) || !aligned16(s_col))))
    return MX_ERR_MISALIGNED;
  DeviceState* st = nullptr;
  mx_status status = device_state(&st);
  if (status != MX_OK) return status;
  mx::QuantizeParams p{};
  p.x = x;
  p.rows = total_rows;
  p.cols = cols;
  p.ldx = ldx;
  p.q_row = row ? q_row : nullptr;
  p.s_row = row ? s_row : nullptr;
  p.q_col = col ? q_col : nullptr;
  p.s_col = col ? s_col : nullptr;
  p.ldq_col = col ? ldq_col : 0;
  p.fmt = fmt;
  p.rule = rule;
  p.offsets = d_offsets;
  p.groups = groups;
  p.status = st->status;
  p.wait_limit_ns = g_wait_ns.load(std::memory_order_relaxed);
  if (cols == 0) return MX_OK;
  if (!all_on_device(st->device, {x, d_offsets, p.q_row, p.s_row, p.q_col, p.s_col}))
    return MX_ERR_INVALID_ARG;
  CUtensorMap tmap;
  // an empty token set still needs a valid map (1 row) for the offsets check
  const int64_t map_rows = total_rows > 0 ? total_rows : 1;
  status = f32 ? encode_f32_map(&tmap, x, cols, map_rows, ldx)
               : encode_bf16_map(&tmap, x, cols, map_rows, ldx);
  if (status != MX_OK) return status;
  const cudaError_t err = f32 ? mx::launch_quantize_grouped_f32(p, tmap, st->num_sms, stream)
                              : mx::launch_quantize_grouped(p, tmap, st->num_sms, stream);
  return err == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

mx_status mx_gemm(int64_t m, int64_t n, int64_t k, const uint8_t* a, const uint8_t* sa, mx_fmt fa,
                  const uint8_t* b, const uint8_t* sb, mx_fmt fb, void* y, mx_dtype y_dtype,
                  int64_t ldy, cudaStream_t stream) {
  return gemm_common(dense_shape(m, n, k), a, sa, fa, b, sb, fb, y, y_dtype, ldy, stream);
}

mx_status mx_gemm_bias_act(int64_t m, int64_t n, int64_t k, const uint8_t* a, const uint8_t* sa,
                           mx_fmt fa, const uint8_t* b, const uint8_t* sb, mx_fmt fb,
                           const float* bias, mx_activation act, void* y, mx_dtype y_dtype,
                           int64_t ldy, cudaStream_t stream) {
  if (act != MX_ACT_NONE && act != MX_ACT_SILU) return MX_ERR_INVALID_ARG;
  if (bias != nullptr && !aligned16(bias)) return MX_ERR_MISALIGNED;
  return gemm_common(dense_shape(m, n, k), a, sa, fa, b, sb, fb, y, y_dtype, ldy, stream, bias,
                     act);
}

mx_status mx_grouped_gemm(int32_t groups, const int32_t* d_offsets, int64_t total_m, int64_t n,
                          int64_t k, const uint8_t* a, const uint8_t* sa, mx_fmt fa,
                          const uint8_t* b, const uint8_t* sb, mx_fmt fb, void* y,
                          mx_dtype y_dtype, cudaStream_t stream) {
  if (groups < 1 || groups > 1000 || !d_offsets) return MX_ERR_INVALID_ARG;
  if (n % 128 != 0) return MX_ERR_INVALID_ARG;
  GemmShape g = dense_shape(total_m, n, k);
  g.b_rows = static_cast<int64_t>(groups) * n;
  g.groups = groups;
  g.d_offsets = d_offsets;
  g.mode = mx::kModeGroupM;
  return gemm_common(g, a, sa, fa, b, sb, fb, y, y_dtype, n, stream);
}

mx_status mx_grouped_gemm_bcat(int32_t groups, const int32_t* d_offsets, int64_t total_m,
                               int64_t n, int64_t k, const uint8_t* a, const uint8_t* sa,
                               mx_fmt fa, const uint8_t* b, int64_t ldb, const uint8_t* sb,
                               mx_fmt fb, void* y, mx_dtype y_dtype, cudaStream_t stream) {
  if (groups < 1 || groups > 1000 || !d_offsets) return MX_ERR_INVALID_ARG;
  if (k <= 0 || k % 128 != 0 || ldb < static_cast<int64_t>(groups) * k) return MX_ERR_INVALID_ARG;
  GemmShape g = dense_shape(total_m, n, k);
  g.ldb = ldb;
  g.b_rows = n;
  g.groups = groups;
  g.d_offsets = d_offsets;
  g.mode = mx::kModeGroupM;
  g.b_concat = 1;
  return gemm_common(g, a, sa, fa, b, sb, fb, y, y_dtype, n, stream);
}

mx_status mx_grouped_gemm_wgrad(int32_t groups, const int32_t* d_offsets, int64_t total_tokens,
                                int64_t m, int64_t n, int64_t ldk, const uint8_t* a,
                                const uint8_t* sa, mx_fmt fa, const uint8_t* b,
                                const uint8_t* sb, mx_fmt fb, void* y, mx_dtype y_dtype,
                                cudaStream_t stream) {
  if (groups < 1 || groups > 1000 || !d_offsets) return MX_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens > INT32_MAX || ldk <= 0 || ldk % 128 != 0)
    return MX_ERR_INVALID_ARG;
  // k carries the token total for the device-side offsets check; each
  // group contracts its own share of the tokens
  GemmShape g;
  g.m = m;
  g.n = n;
  g.k = total_tokens;
  g.lda = ldk;
  g.ldb = ldk;
  g.b_rows = n;
  g.groups = groups;
  g.d_offsets = d_offsets;
  g.mode = mx::kModeGroupK;
  return gemm_common(g, a, sa, fa, b, sb, fb, y, y_dtype, n, stream);
}

mx_status mx_device_status(cudaStream_t stream) {
  DeviceState* st = nullptr;
  mx_status s = device_state(&st);
  if (s != MX_OK) return s;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MX_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, st->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MX_ERR_CUDA;
  if (word != 0) {
    // clear only the bits read here (a kernel on another stream may set one
    // meanwhile; it then stays for the next query)
    if (mx::launch_status_clear(st->status, word, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return MX_ERR_CUDA;
  }
  if (word & 1u) return MX_ERR_TIMEOUT;
  if (word & 2u) return MX_ERR_DEVICE_ARG;
  return MX_OK;
}

mx_status mx_set_wait_timeout_ns(uint64_t ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
  return MX_OK;
}

mx_status mx_selftest_wait_timeout(uint64_t ns, cudaStream_t stream) {
  if (ns == 0 || ns > 10000000000ull) return MX_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  mx_status s = device_state(&st);
  if (s != MX_OK) return s;
  return mx::launch_wait_selftest(st->status, ns, stream) == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

const char* mx_status_str(mx_status status) {
  switch (status) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
    case MX_ERR_MISALIGNED: return "MX_ERR_MISALIGNED";
    case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
    case MX_ERR_CUDA: return "MX_ERR_CUDA";
    case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT";
    case MX_ERR_DEVICE_ARG: return "MX_ERR_DEVICE_ARG";
  }
  return "MX_ERR_UNKNOWN";
}

}  // extern "C"
