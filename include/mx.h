/*
 * mx.h -- C ABI of libmx, the MXFP8 training-matmul library for GB300 (sm_103a).
 *
 * The library has two parts, after "Low-Precision GPU Programming"
 * (leetllm.com):
 *
 *   1. MX quantization (sections "Format taxonomy: range, spacing, and
 *      bitfields", "Numerical hazards: subnormals, saturation, and rounding"
 *      and "Microscaling: the two-row experiment"): every block of 32
 *      consecutive elements along the contraction axis K shares one E8M0
 *      power-of-two scale S, and each element becomes the OCP E4M3 or E5M2
 *      code of x / S, rounded to nearest even with saturation to the finite
 *      range.
 *   2. The block-scaled GEMM (section "Scale ownership and the GEMM
 *      dataflow"): Y[i,j] = sum_b S_A[i,b] * S_B[j,b] * sum_{k in b}
 *      A~[i,k] * B~[j,k], accumulated in FP32 on the tensor cores, with an
 *      epilogue that writes FP32 or BF16 (round to nearest even).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers marked "device" must point to device memory of the current
 *    CUDA device (memory of cudaMalloc or of a memory pool on that device);
 *    the caller allocates and owns every buffer.  Every entry point checks
 *    this with cudaPointerGetAttributes and returns MX_ERR_INVALID_ARG,
 *    launching nothing, for host memory (pageable, pinned or mapped),
 *    managed memory or another device's memory.  The library allocates no
 *    device memory.
 *  - Work is enqueued on `stream` (0 = legacy default stream).  No entry
 *    point synchronizes the stream or the device (except mx_device_status),
 *    and none keeps per-call device scratch, so the calls may be captured
 *    into CUDA graphs and issued on several streams and from several host
 *    threads concurrently.
 *  - Arguments are validated on the host before anything is launched; a
 *    non-MX_OK status means nothing was enqueued.
 *  - Faults detected on the device (a pipeline wait that timed out, invalid
 *    group offsets) are recorded in one status word per device, shared by
 *    every stream and host thread of the process, and reported by
 *    mx_device_status().  A fault of a kernel on any stream is therefore
 *    reported to whichever caller queries the device first.
 *  - Every device pointer must be 16-byte aligned, and every leading
 *    dimension must span a multiple of 16 bytes (MX_ERR_MISALIGNED).
 *  - Sizes: rows, K and leading dimensions up to 2^31 - 1; a GEMM whose
 *    256x256 output tiles (over all groups) number 2^31 or more, and a
 *    quantization whose (padded) tiles of 128 rows x 128 bf16 or 64 FP32
 *    columns number 2^32 or more, return MX_ERR_UNSUPPORTED.
 *
 * Scale layout ("swizzled", the operand layout of the tensor-core
 * block-scaled MMA; the pages require the layout to be recorded with the
 * kernel but do not define it -- section "Hardware support and kernel ABI
 * contracts"):
 *  - Scales of a [rows, K] operand (ceil(K/32) blocks per row; a final
 *    block of K % 32 elements is the page's zero-padded partial block) are
 *    stored in tiles
 *    of 128 rows x 4 blocks = 512 bytes.  Tile (rt, kt) starts at byte
 *    (rt * ceil(K/128) + kt) * 512.  Inside a tile, the scale of local row r
 *    (0..127) and local block c (0..3) is at byte
 *    (r % 32) * 16 + (r / 32) * 4 + c.
 *  - Padding entries (rows >= rows, blocks >= ceil(K/32)) are written as 0x00 by
 *    the quantizer and never influence a valid GEMM output.
 *  - A scale byte c encodes 2^(c - 127); 0xFF is NaN.
 *
 * Kernels: quantization runs in one persistent kernel (one block per SM,
 * tiles streamed by TMA); every GEMM runs in one block-pair kernel
 * (tcgen05 cta_group::2, 256x256 output tiles over two SMs).  No
 * environment variable changes what the library does.
 */
#ifndef MX_H_
#define MX_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MX_OK = 0,
  MX_ERR_INVALID_ARG = 1,   /* shape, enum or null-pointer error              */
  MX_ERR_MISALIGNED = 2,    /* pointer or leading dimension not 16-byte aligned */
  MX_ERR_UNSUPPORTED = 3,   /* valid but not implemented combination          */
  MX_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed            */
  MX_ERR_TIMEOUT = 5,       /* a device pipeline wait gave up (device status) */
  MX_ERR_DEVICE_ARG = 6     /* the device found invalid data (group offsets)  */
} mx_status;

/* Element formats, section "Format taxonomy: range, spacing, and
 * bitfields".  FP8 (OCP OFP8): E4M3 max 448, no Inf, NaN 0x7F/0xFF; E5M2
 * max 57344, IEEE-like Inf and NaN.  MXFP6: E2M3 (max 7.5) and E3M2 (max
 * 28); MXFP4: E2M1 (max 6); these three have no Inf or NaN encodings.
 * FP8 codes are one byte per element.  The 6- and 4-bit codes come in two
 * storage layouts:
 *  - MX_E2M3, MX_E3M2, MX_E2M1: the tensor-core container layout: every run
 *    of 16 elements along K occupies 16 bytes, the 16 codes packed
 *    little-endian (element i at bits [i*w, i*w + w) of the run, w = 6 or
 *    4) followed by zero bytes -- a code buffer has the size and strides of
 *    an FP8 one (one byte per element).
 *  - MX_E2M3_PACKED, MX_E3M2_PACKED, MX_E2M1_PACKED: the same codes densely
 *    packed, the payload the page counts for narrow elements: a row of K
 *    elements is one little-endian bit string of K*w/8 bytes, element i at
 *    bits [i*w, i*w + w) (E2M1: two codes per byte, element 2i in the low
 *    nibble; E2M3 and E3M2: four codes per three bytes).  The GEMM reads
 *    them with the tensor copy's unpacking element types, which place each
 *    16-element run in the container layout in shared memory.  A GEMM
 *    operand in packed storage needs K % 128 == 0 and a 32-byte aligned code
 *    pointer. */
typedef enum {
  MX_E4M3 = 0, MX_E5M2 = 1, MX_E2M3 = 2, MX_E3M2 = 3, MX_E2M1 = 4,
  MX_E2M3_PACKED = 5, MX_E3M2_PACKED = 6, MX_E2M1_PACKED = 7
} mx_fmt;

/* Wide element types: quantizer input (bf16 or FP32, both taken exactly:
 * every input value is representable, so the block amax, the scale and the
 * one rounding to the element grid are those of the exact value) and GEMM
 * output. */
typedef enum { MX_BF16 = 0, MX_FP32 = 1 } mx_dtype;

/* Which quantizations to produce from one read of the wide tensor.
 * ROWWISE: 1x32 blocks along the columns of x.  COLWISE: 32x1 blocks along
 * the rows of x, written transposed so that the blocked axis is contiguous.
 * (section "Microscaling: the two-row experiment": both orientations are
 * derived from the original wide data, never by moving codes.) */
typedef enum { MX_ROWWISE = 1, MX_COLWISE = 2, MX_BOTH = 3 } mx_axis;

/* Block scale rule.
 * MX_SCALE_FLOOR: S = 2^(floor(log2 amax) - emax_elem), emax_elem = 8 for
 *   E4M3 and 15 for E5M2 (the OCP MX rule); values above the format maximum
 *   after scaling saturate.
 * MX_SCALE_CEIL: S = 2^ceil(log2(amax / max)), the conservative rule the
 *   two-row experiment uses; no element saturates.
 * Both: exponent clamped to [-127, 127]; an all-zero block takes S = 1; a
 * block holding NaN or Inf takes scale 0xFF and, for every element, the NaN
 * code 0x7F of E4M3 / E5M2, or code 0 for E2M3, E3M2 and E2M1 (which have
 * no NaN encoding).  MX_SCALE_CEIL is the rule some documents call RCEIL
 * ("round the scale up"); with amax = m * 2^E, m in [1, 2), it equals the
 * floor rule's exponent plus one exactly when m exceeds the significand of
 * the format's maximum (1.75 for E4M3, E5M2 and E3M2; 1.875 for E2M3; 1.5
 * for E2M1). */
typedef enum { MX_SCALE_FLOOR = 0, MX_SCALE_CEIL = 1 } mx_scale_rule;

/* Bytes of the swizzled scale buffer of a [rows, k] operand:
 * ceil(rows/128)*128 * ceil(ceil(k/32)/4)*4.  k must be a multiple of 16
 * (returns 0 otherwise or for negative sizes). */
size_t mx_scale_bytes(int64_t rows, int64_t k);

/* Upper bound of the per-group padded scale buffer used by
 * mx_quantize_grouped / mx_grouped_gemm for any split of total_rows into
 * `groups` groups: (ceil(total_rows/128) + groups) * 128 * ceil(k/128) * 4. */
size_t mx_grouped_scale_bytes(int64_t total_rows, int32_t groups, int64_t k);

/* MX quantization of a bf16 or FP32 matrix x[rows, cols] (x_dtype;
 * row-major, leading dimension ldx elements), section "Microscaling: the
 * two-row experiment".
 *
 *  ROWWISE (needs cols % 16 == 0): q_row[rows, cols] codes (row-major,
 *    leading dimension cols) and s_row = swizzled scales of the
 *    [rows, cols] operand (mx_scale_bytes(rows, cols) bytes).
 *  COLWISE (needs rows % 16 == 0): q_col[cols, rows] codes -- the transpose,
 *    leading dimension rows -- and s_col = swizzled scales of the
 *    [cols, rows] operand (mx_scale_bytes(cols, rows) bytes).
 *  Blocked axis not a multiple of 32: the final block holds 16 elements
 *    and is quantized as the zero-padded partial block of section "Scale
 *    ownership and the GEMM dataflow" (its amax and scale are those of its
 *    16 elements; no code is written past the matrix).  Packed formats
 *    need the blocked axis % 32 == 0.
 *  BOTH: both of the above from one read of x.
 *  Packed formats (MX_*_PACKED): a code row of n elements takes n*w/8 bytes
 *    (q_row: rows x cols*w/8 bytes; q_col: cols x rows*w/8 bytes).
 *
 * x, q_*, s_* are device pointers; unused outputs may be NULL.
 * cols % 8 == 0, ldx >= cols, and rows of x start on 16-byte boundaries:
 * ldx % 8 == 0 for MX_BF16, ldx % 4 == 0 for MX_FP32 (else
 * MX_ERR_MISALIGNED); another x_dtype is MX_ERR_INVALID_ARG.
 * Codes and scales are bit-exact functions of x (no rounding-order freedom). */
mx_status mx_quantize(const void* x, mx_dtype x_dtype, int64_t rows, int64_t cols,
                      int64_t ldx, mx_fmt fmt, mx_axis axis, mx_scale_rule rule,
                      uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                      cudaStream_t stream);

/* mx_quantize with stochastic rounding in place of round-to-nearest-even
 * (section "Rounding: RNE versus stochastic rounding").  rbits: device
 * uint16[rows, cols] (leading dimension ldr elements, ldr % 8 == 0), one
 * random integer r per element of x, used by both orientations.  With l <= |v|
 * < u the neighbouring grid values of the exactly scaled element v, |v| goes
 * to u iff r < floor(2^16 (|v| - l) / (u - l)), else to l; the result then
 * saturates like the RNE path.  Scales are those of mx_quantize (they depend
 * only on the block amax).  Every element format and storage of mx_quantize
 * is accepted (FP8, and the 6- and 4-bit codes in the container or packed
 * storage).  For a given rbits the codes are bit-exact. */
mx_status mx_quantize_sr(const void* x, mx_dtype x_dtype, int64_t rows, int64_t cols,
                         int64_t ldx, const uint16_t* rbits, int64_t ldr, mx_fmt fmt,
                         mx_axis axis, mx_scale_rule rule,
                         uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                         cudaStream_t stream);

/* Rowwise MX quantization of routed tokens x[total_rows, cols] grouped by
 * expert: rows [d_offsets[g], d_offsets[g+1]) belong to group g.  Codes are
 * written as by mx_quantize ROWWISE; scales use the per-group padded layout
 * that mx_grouped_gemm reads: group g's scales form their own swizzled
 * matrix starting at row P_g = sum_{h<g} ceil(m_h/128)*128, i.e. at byte
 * (P_g/128) * ceil(cols/128) * 512.  s must hold
 * mx_grouped_scale_bytes(total_rows, groups, cols) bytes; bytes past the
 * last group are left untouched.  d_offsets: device int32[groups + 1],
 * d_offsets[0] = 0, non-decreasing, d_offsets[groups] = total_rows; invalid
 * offsets are reported through mx_device_status (MX_ERR_DEVICE_ARG) and
 * nothing is written.  1 <= groups <= 1000.  x_dtype and ldx as for
 * mx_quantize; fmt MX_E4M3 or MX_E5M2 (other formats MX_ERR_UNSUPPORTED). */
mx_status mx_quantize_grouped(const void* x, mx_dtype x_dtype, int64_t total_rows,
                              int64_t cols, int64_t ldx, mx_fmt fmt, mx_scale_rule rule,
                              int32_t groups, const int32_t* d_offsets,
                              uint8_t* q, uint8_t* s, cudaStream_t stream);

/* Upper bound of the token columns that the per-group padded columnwise
 * layout of mx_quantize_grouped_ex needs for any split of total_rows into
 * `groups` groups: 128 * (floor(total_rows / 128) + groups) (each group
 * rounds its token count up to a multiple of 128).  0 for negative input. */
int64_t mx_grouped_cols_capacity(int64_t total_rows, int32_t groups);

/* MX quantization of routed tokens x[total_rows, cols] grouped by expert,
 * in either or both orientations from one read (axis).
 * ROWWISE: exactly mx_quantize_grouped (q_row, s_row).
 * COLWISE: per group g, the 32-row blocks start at the group's first row
 *   (no block spans two groups) and a final partial block is completed with
 *   zeros -- the zero-padded final block of section "Scale ownership and
 *   the GEMM dataflow".  The transposed codes of all groups share one
 *   q_col[cols, ldq_col] matrix (K = tokens, contiguous): group g occupies
 *   columns [P_g, P_g + ceil(m_g/128)*128), P_g = sum_{h<g} ceil(m_h/128)*128,
 *   padding tokens holding code 0; s_col holds the swizzled scales of the
 *   whole [cols, ldq_col] operand (mx_scale_bytes(cols, ldq_col) bytes),
 *   padding blocks 0.  Columns past the last group are left untouched.
 *   ldq_col % 128 == 0 and ldq_col >= P_groups (mx_grouped_cols_capacity
 *   always suffices); a layout that does not fit is reported through
 *   mx_device_status (MX_ERR_DEVICE_ARG) and nothing is written.  This is
 *   the operand layout of mx_grouped_gemm_wgrad.
 * cols % 8 == 0 (ROWWISE also cols % 16 == 0); x_dtype, ldx, d_offsets and
 * groups as for mx_quantize and mx_quantize_grouped.  Unused outputs may be
 * NULL. */
mx_status mx_quantize_grouped_ex(const void* x, mx_dtype x_dtype, int64_t total_rows,
                                 int64_t cols, int64_t ldx, mx_fmt fmt, mx_axis axis,
                                 mx_scale_rule rule, int32_t groups, const int32_t* d_offsets,
                                 uint8_t* q_row, uint8_t* s_row,
                                 uint8_t* q_col, int64_t ldq_col, uint8_t* s_col,
                                 cudaStream_t stream);

/* Block-scaled GEMM, section "Scale ownership and the GEMM dataflow":
 *   y[i, j] = sum_b S_A[i,b] S_B[j,b] sum_{k in b} A~[i,k] B~[j,k]
 * A: a[m, k] codes (row-major, K contiguous, leading dimension k) with
 *    swizzled scales sa of the [m, k] operand -- e.g. X quantized ROWWISE.
 * B: b[n, k] codes (K contiguous, leading dimension k) with swizzled scales
 *    sb of the [n, k] operand -- e.g. W[k, n] quantized COLWISE (= W^T).
 * fa, fb: any element format of mx_fmt, in any combination; 6- and 4-bit
 *    codes in either storage layout described with mx_fmt (packed storage:
 *    k % 128 == 0, code pointer 32-byte aligned, row stride k*w/8 bytes).
 * y: device, [m, n] row-major with leading dimension ldy (elements),
 *    FP32 or BF16 (RNE from the FP32 accumulator).
 * Constraints: k % 16 == 0, k >= 16, n % 8 == 0, ldy >= n.  When k % 32 ==
 * 16 the final block is the zero-padded partial block (codes past k read as
 * zero; its scales are those mx_quantize writes for it).
 * Accumulation is FP32 on the tensor cores; its internal order is
 * implementation-defined (section "Accumulator type isn't the whole
 * arithmetic contract"). */
mx_status mx_gemm(int64_t m, int64_t n, int64_t k,
                  const uint8_t* a, const uint8_t* sa, mx_fmt fa,
                  const uint8_t* b, const uint8_t* sb, mx_fmt fb,
                  void* y, mx_dtype y_dtype, int64_t ldy, cudaStream_t stream);

/* Activation of the fused epilogue. */
typedef enum { MX_ACT_NONE = 0, MX_ACT_SILU = 1 } mx_activation;

/* mx_gemm with the fused epilogue of the kernel contract in section
 * "Hardware support and kernel ABI contracts" (FP32 bias, SiLU, BF16 out):
 *   y[i, j] = act(acc[i, j] + bias[j]),  act(z) = z / (1 + exp(-z)) for SiLU
 * The bias add and the activation run in FP32 on the FP32 accumulator,
 * followed by one rounding to y_dtype (RNE for BF16).
 * bias: device float[n], 16-byte aligned, or NULL for no bias.
 * act: MX_ACT_NONE or MX_ACT_SILU.  Other arguments and constraints as
 * mx_gemm. */
mx_status mx_gemm_bias_act(int64_t m, int64_t n, int64_t k,
                           const uint8_t* a, const uint8_t* sa, mx_fmt fa,
                           const uint8_t* b, const uint8_t* sb, mx_fmt fb,
                           const float* bias, mx_activation act,
                           void* y, mx_dtype y_dtype, int64_t ldy, cudaStream_t stream);

/* Grouped (mixture-of-experts) block-scaled GEMM: for every group g,
 *   y[o_g : o_{g+1}, :] = A[o_g : o_{g+1}, :] * B_g^T
 * with the per-row block scales of the dense GEMM.
 * a: [total_m, k] codes of the concatenated tokens; sa: per-group padded
 *    swizzled scales (as written by mx_quantize_grouped).
 * b: [groups, n, k] codes (each B_g K-contiguous); sb: groups consecutive
 *    swizzled scale matrices of [n, k], group g at byte g * mx_scale_bytes(n, k).
 * y: [total_m, n] row-major (leading dimension n).  Rows of empty groups do
 *    not exist; rows outside [0, total_m) are never written.
 * d_offsets: device int32[groups + 1] as for mx_quantize_grouped; read on
 *    the device (no host synchronization).  n % 128 == 0, k % 16 == 0. */
mx_status mx_grouped_gemm(int32_t groups, const int32_t* d_offsets, int64_t total_m,
                          int64_t n, int64_t k,
                          const uint8_t* a, const uint8_t* sa, mx_fmt fa,
                          const uint8_t* b, const uint8_t* sb, mx_fmt fb,
                          void* y, mx_dtype y_dtype, cudaStream_t stream);

/* Grouped GEMM with the experts' B operands side by side along K (the
 * data-gradient GEMM of a mixture of experts, dX_g = dY_g W_g^T):
 *   y[o_g : o_{g+1}, :] = A[o_g : o_{g+1}, :] * B_g^T,  B_g = b[:, g*k : (g+1)*k]
 * a, sa, d_offsets, y: as for mx_grouped_gemm (a: [total_m, k] rowwise,
 *    per-group padded scales).
 * b: one [n, ldb] code matrix (K contiguous) with swizzled scales sb of the
 *    whole [n, ldb] operand -- exactly what mx_quantize COLWISE writes for
 *    the stacked expert weights viewed as [groups * k, n] (e.g. W^T of every
 *    expert stored [groups, k, n]); 32-row blocks never span two experts
 *    because k % 32 == 0.
 * Constraints: k % 128 == 0 (each expert starts on a scale tile),
 * ldb >= groups * k, ldb % 16 == 0, n % 8 == 0. */
mx_status mx_grouped_gemm_bcat(int32_t groups, const int32_t* d_offsets, int64_t total_m,
                               int64_t n, int64_t k,
                               const uint8_t* a, const uint8_t* sa, mx_fmt fa,
                               const uint8_t* b, int64_t ldb, const uint8_t* sb, mx_fmt fb,
                               void* y, mx_dtype y_dtype, cudaStream_t stream);

/* Per-expert weight gradient of a mixture of experts, a GEMM grouped along
 * its contraction: for every group g with m_g = o_{g+1} - o_g tokens,
 *   y[g] = A_g * B_g^T,  A_g = a[:, P_g : P_g + m_g],  B_g = b[:, P_g : P_g + m_g]
 * contracted over that expert's tokens only (section "Scale ownership and
 * the GEMM dataflow", with the final partial block zero-padded).
 * a: [m, ldk] codes with swizzled scales sa of the [m, ldk] operand;
 *    b: [n, ldk] likewise -- both as written by mx_quantize_grouped_ex
 *    COLWISE with the same d_offsets and ldk (e.g. a from dY[tokens, m],
 *    b from X[tokens, n], giving y[g] = dY_g^T X_g).
 * y: [groups, m, n] row-major (group g at element g*m*n); an expert without
 *    tokens gets zeros.
 * d_offsets: device int32[groups + 1], 0 = o_0 <= ... <= o_groups =
 *    total_tokens, read on the device; invalid offsets, or segments that do
 *    not fit in ldk, are reported through mx_device_status
 *    (MX_ERR_DEVICE_ARG) and nothing is written.
 * Constraints: ldk % 128 == 0, n % 8 == 0, 1 <= groups <= 1000. */
mx_status mx_grouped_gemm_wgrad(int32_t groups, const int32_t* d_offsets, int64_t total_tokens,
                                int64_t m, int64_t n, int64_t ldk,
                                const uint8_t* a, const uint8_t* sa, mx_fmt fa,
                                const uint8_t* b, const uint8_t* sb, mx_fmt fb,
                                void* y, mx_dtype y_dtype, cudaStream_t stream);

/* Synchronizes `stream`, then reads the device status word of the current
 * device and clears the bits it read: MX_OK, MX_ERR_TIMEOUT (a kernel's
 * bounded pipeline wait gave up; its outputs are undefined) or
 * MX_ERR_DEVICE_ARG (invalid group offsets).  The word is shared by all
 * streams of the device, so the fault may come from a kernel on another
 * stream; a bit that such a kernel sets after the read stays set for the
 * next call.  MX_ERR_CUDA if the synchronization itself failed. */
mx_status mx_device_status(cudaStream_t stream);

/* Static string naming a status code. */
const char* mx_status_str(mx_status status);

/* Bounded pipeline waits: every mbarrier wait inside the kernels gives up
 * after `ns` nanoseconds (default 2e9 when ns == 0), records MX_ERR_TIMEOUT
 * in the device status word and lets the kernel drain and exit.  Applies to
 * launches enqueued after the call, on every device. */
mx_status mx_set_wait_timeout_ns(uint64_t ns);

/* Self-test of the bounded wait: enqueues one tiny kernel that waits on an
 * mbarrier that nothing ever completes, with a limit of `ns` nanoseconds.
 * mx_device_status() afterwards must return MX_ERR_TIMEOUT.  No TMA, MMA or
 * tensor memory is involved. */
mx_status mx_selftest_wait_timeout(uint64_t ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MX_H_ */
