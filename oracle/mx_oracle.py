"""CPU oracle for MXFP8 training matmul: quantization and block-scaled GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code, table or
constant with the CUDA library in ``mxfp8_block_scaled_mx_gb300/csrc``.

Every function is the plain definition written out in float64 / Python
integers, with no blocking, fusion or reordering beyond what the definition
states.  Sources (page title, section):

* "Low-Precision GPU Programming" (leetllm.com), section "Format taxonomy:
  range, spacing, and bitfields" -- OCP E4M3 / E5M2 ranges, NaN codes,
  grid spacing, and the MX block of 32 elements with one E8M0 scale.
* same page, "Numerical hazards: subnormals, saturation, and rounding" --
  round-to-nearest-even including subnormals and signed zero; saturating
  conversion rounds first, then limits the magnitude to the format maximum.
* same page, "One letter, two reciprocal conventions" -- S is the
  reconstruction scale: x_hat = S * q and q = Q(x / S); a zero-only group
  takes S = 1.
* same page, "Microscaling: the two-row experiment" -- E8M0 byte c in
  [0, 254] is 2^(c - 127), 255 is NaN; the conservative power-of-two rule
  S = 2^ceil(log2(amax / max)) with the exponent clamped at -127.
* same page, "Scale ownership and the GEMM dataflow" -- with 32-element
  blocks along K the block scale product stays inside the outer sum:
  Y_ij = sum_b S_X[i,b] * S_W[b,j] * sum_{k in b} Xq[i,k] * Wq[k,j],
  a partial final block (K not a multiple of 32) completed with zeros.
* same page, "Hardware support and kernel ABI contracts" -- the kernel
  contract's epilogue: an FP32 bias per output column, then SiLU, then BF16.
  SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)).
* The MX block scale rule used by the product (the "floor" rule of the OCP
  MX specification):
  S = 2^(floor(log2 amax) - emax_elem), emax_elem = 8 (E4M3) or 15 (E5M2).

Readings where the pages are silent:

* A block holding NaN or +-Inf gets scale byte 0xFF (NaN) and every code in
  it is the NaN code 0x7F.
* E5M2 special values follow the IEEE pattern: exponent field 31 with
  mantissa 0 is Inf, otherwise NaN.
* Scale exponents are clamped to [-127, 127] (E8M0 has no code below 0).
* The swizzled scale layout is the one the Blackwell block-scaled tensor-core
  MMA consumes (128-row x 4-block tiles of 512 bytes; see ``swizzle_offset``).
  The pages do not define it.  parity unpinned on the CPU: the layout is
  pinned only by the tensor core consuming bytes written by this module.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from fractions import Fraction

import numpy as np

# --------------------------------------------------------------------------
# Element formats
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class Fp8Format:
    """An OCP element format: sign, ebits exponent bits, mbits mantissa bits
    (FP8, and the narrower MXFP6 / MXFP4 element formats)."""
    name: str
    ebits: int       # exponent field width
    mbits: int       # mantissa field width
    bias: int
    emax_elem: int   # exponent of the largest binade (floor(log2(max)))
    max_finite: float
    has_inf: bool
    has_nan: bool = True

    @property
    def bits(self) -> int:
        return 1 + self.ebits + self.mbits

    @property
    def min_normal(self) -> float:
        return 2.0 ** (1 - self.bias)

    @property
    def subnormal_step(self) -> float:
        return 2.0 ** (1 - self.bias - self.mbits)

    @property
    def nan_code(self) -> int:
        """Code written for every element of a NaN/Inf block: the FP8 NaN
        0x7F; formats without NaN encodings write 0 (the block's NaN scale
        alone marks it)."""
        return NAN_CODE if self.has_nan else 0


# OCP E4M3: bias 7, max 448 = 1.75 * 2^8, no Inf, NaN at S.1111.111.
E4M3 = Fp8Format("e4m3", 4, 3, 7, 8, 448.0, False)
# OCP E5M2: bias 15, max 57344 = 1.75 * 2^15, IEEE-like Inf / NaN.
E5M2 = Fp8Format("e5m2", 5, 2, 15, 15, 57344.0, True)
# OCP MX element formats without Inf or NaN ("Format taxonomy": MXFP6 uses
# E3M2, maximum 28, or E2M3, maximum 7.5; MXFP4 uses E2M1, maximum 6).
E2M3 = Fp8Format("e2m3", 2, 3, 1, 2, 7.5, False, False)
E3M2 = Fp8Format("e3m2", 3, 2, 3, 4, 28.0, False, False)
E2M1 = Fp8Format("e2m1", 2, 1, 1, 2, 6.0, False, False)
FORMATS = {"e4m3": E4M3, "e5m2": E5M2, "e2m3": E2M3, "e3m2": E3M2, "e2m1": E2M1}

NAN_CODE = 0x7F          # canonical NaN code emitted for NaN/Inf blocks (FP8)
E8M0_NAN = 0xFF


def fmt_of(f) -> Fp8Format:
    return f if isinstance(f, Fp8Format) else FORMATS[f]


# --------------------------------------------------------------------------
# Decoding
# --------------------------------------------------------------------------


def decode_code(fmt, code: int) -> float:
    """Value of one code (float64; exact, the grid is dyadic).  The sign is
    the top bit of the format's width."""
    f = fmt_of(fmt)
    if not 0 <= code < (1 << f.bits):
        raise ValueError("code out of range")
    sign = -1.0 if code >> (f.bits - 1) else 1.0
    e = (code >> f.mbits) & ((1 << f.ebits) - 1)
    m = code & ((1 << f.mbits) - 1)
    e_all_ones = (1 << f.ebits) - 1
    if f.has_inf:
        if e == e_all_ones:
            return sign * math.inf if m == 0 else math.nan
    elif f.has_nan and e == e_all_ones and m == (1 << f.mbits) - 1:
        return math.nan
    if e == 0:
        return sign * (m / (1 << f.mbits)) * 2.0 ** (1 - f.bias)
    return sign * (1.0 + m / (1 << f.mbits)) * 2.0 ** (e - f.bias)


def decode_table(fmt) -> np.ndarray:
    """float64[2^bits]: value of every code."""
    f = fmt_of(fmt)
    return np.array([decode_code(f, c) for c in range(1 << f.bits)], dtype=np.float64)


def decode_e8m0(code: int) -> float:
    """E8M0 scale byte: 2^(code - 127) for 0..254, NaN for 255."""
    if not 0 <= code <= 255:
        raise ValueError("scale byte out of range")
    return math.nan if code == E8M0_NAN else 2.0 ** (code - 127)


def e8m0_values(scales: np.ndarray) -> np.ndarray:
    s = scales.astype(np.int64)
    out = np.ldexp(1.0, s - 127).astype(np.float64)
    out[s == E8M0_NAN] = np.nan
    return out


# --------------------------------------------------------------------------
# Encoding: round to nearest even on the format grid, then saturate
# --------------------------------------------------------------------------


def round_to_grid_rne(fmt, v: np.ndarray) -> np.ndarray:
    """Nearest grid value of |v| (ties to even significand), sign restored.

    The grid is the format's finite values extended past the maximum with the
    top binade's spacing; no saturation here.  Inputs must be finite.
    """
    f = fmt_of(fmt)
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    # quantum (grid spacing) at |v|: subnormal spacing below the smallest
    # normal, else 2^(floor(log2|v|) - mbits).
    _, ex = np.frexp(a)                      # a = frac * 2^ex, frac in [0.5, 1)
    floor_log2 = ex.astype(np.int64) - 1
    quantum_exp = np.where(a < f.min_normal, 1 - f.bias - f.mbits,
                           floor_log2 - f.mbits)
    # a / quantum and n * quantum are exact (powers of two, no over/underflow
    # for float64 inputs in the ranges used here); np.rint rounds half to even.
    n = np.rint(np.ldexp(a, -quantum_exp))
    r = np.ldexp(n, quantum_exp)
    return np.copysign(r, v)


SR_BITS = 16


def round_to_grid_stochastic(fmt, v: np.ndarray, rand: np.ndarray) -> np.ndarray:
    """Stochastic rounding ("Rounding: RNE versus stochastic rounding"): with
    l <= |v| < u the neighbouring grid values (grid extended past the
    maximum, no saturation here), |v| goes to u with probability
    frac = (|v| - l) / (u - l), else to l; sign restored.  Reading: the random
    draw is an input integer r in [0, 2^16) per element, and |v| goes up iff
    r < floor(frac * 2^16) (exact for every frac with at most 16 bits; a
    fraction below 2^-16 of a step never rounds up)."""
    f = fmt_of(fmt)
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)
    floor_log2 = ex.astype(np.int64) - 1
    quantum_exp = np.where(a < f.min_normal, 1 - f.bias - f.mbits, floor_log2 - f.mbits)
    units = np.ldexp(a, -quantum_exp)            # exact: |v| in grid steps
    low = np.floor(units)
    frac16 = np.floor((units - low) * 2.0 ** SR_BITS)
    up = np.asarray(rand, dtype=np.int64) < frac16
    r = np.ldexp(low + up, quantum_exp)
    return np.copysign(r, v)


def encode_sat_sr(fmt, v: np.ndarray, rand: np.ndarray) -> np.ndarray:
    """Saturating stochastic-rounding conversion: round as above, then give
    +-max when the rounded magnitude exceeds it; NaN gives 0x7F."""
    f = fmt_of(fmt)
    v = np.asarray(v, dtype=np.float64)
    nan = np.isnan(v)
    finite_v = np.where(np.isfinite(v), v, np.copysign(2.0 * f.max_finite, v))
    finite_v = np.where(nan, 0.0, finite_v)
    r = round_to_grid_stochastic(f, finite_v, rand)
    r = np.where(np.abs(r) > f.max_finite, np.copysign(f.max_finite, r), r)
    codes = encode_grid_value(f, r)
    codes[nan] = f.nan_code
    return codes


def encode_grid_value(fmt, r: np.ndarray) -> np.ndarray:
    """Bit pattern of exact finite grid values r (|r| <= max)."""
    f = fmt_of(fmt)
    r = np.asarray(r, dtype=np.float64)
    sign = np.signbit(r).astype(np.int64)
    a = np.abs(r)
    _, ex = np.frexp(a)
    floor_log2 = ex.astype(np.int64) - 1
    normal = a >= f.min_normal
    e_field = np.where(normal, floor_log2 + f.bias, 0)
    # mantissa: normal a = (1 + m/2^mbits) 2^(E-bias); subnormal a = m * step
    m_norm = np.ldexp(a, -floor_log2) - 1.0
    m_field = np.where(normal, np.ldexp(m_norm, f.mbits),
                       np.ldexp(a, -(1 - f.bias - f.mbits)))
    m_field = np.where(a == 0, 0.0, m_field)
    m_int = m_field.astype(np.int64)
    assert np.all(m_int == m_field), "value is not on the format grid"
    code = (sign << (f.bits - 1)) | (e_field << f.mbits) | m_int
    return code.astype(np.uint8)


def encode_sat_rne(fmt, v: np.ndarray) -> np.ndarray:
    """Saturating RNE conversion of exact float64 values to element codes.

    Round first; if the rounded magnitude exceeds the maximum finite value,
    give the maximum with the input's sign.  +-Inf saturates likewise, NaN
    gives the format's NaN code (0x7F for FP8, 0 for the formats without
    NaN).  A negative value that rounds to zero gives -0.
    """
    f = fmt_of(fmt)
    v = np.asarray(v, dtype=np.float64)
    nan = np.isnan(v)
    finite_v = np.where(np.isfinite(v), v, np.copysign(2.0 * f.max_finite, v))
    finite_v = np.where(nan, 0.0, finite_v)
    r = round_to_grid_rne(f, finite_v)
    r = np.where(np.abs(r) > f.max_finite, np.copysign(f.max_finite, r), r)
    codes = encode_grid_value(f, r)
    codes[nan] = f.nan_code
    return codes


# --------------------------------------------------------------------------
# MX block scales
# --------------------------------------------------------------------------

BLOCK = 32


def floor_log2_exact(a: np.ndarray) -> np.ndarray:
    """floor(log2 a) for positive finite float64 a (exact, via frexp)."""
    _, ex = np.frexp(a)
    return ex.astype(np.int64) - 1


def scale_exponent_floor(fmt, amax: np.ndarray) -> np.ndarray:
    """OCP MX rule: e = floor(log2 amax) - emax_elem, clamped to [-127, 127].

    amax == 0 takes S = 1 (e = 0).  Caller handles non-finite amax.
    """
    f = fmt_of(fmt)
    amax = np.asarray(amax, dtype=np.float64)
    pos = amax > 0
    e = np.where(pos, floor_log2_exact(np.where(pos, amax, 1.0)) - f.emax_elem, 0)
    return np.clip(e, -127, 127)


def scale_exponent_ceil(fmt, amax: np.ndarray) -> np.ndarray:
    """Conservative rule of the two-row experiment: smallest e with
    amax <= max * 2^e (i.e. e = ceil(log2(amax / max))), clamped below at -127;
    amax == 0 takes S = 1."""
    f = fmt_of(fmt)
    amax = np.asarray(amax, dtype=np.float64)
    pos = amax > 0
    safe = np.where(pos, amax, 1.0)
    e = floor_log2_exact(safe) - floor_log2_exact(np.array(f.max_finite))
    # e is within one of the answer; settle it with exact comparisons
    e = np.where(safe > np.ldexp(f.max_finite, e), e + 1, e)
    e = np.where(safe <= np.ldexp(f.max_finite, e - 1), e - 1, e)
    e = np.where(pos, e, 0)
    return np.clip(e, -127, 127)


def pad_final_block(x: np.ndarray) -> np.ndarray:
    """x[rows, K] completed with zero columns to a whole number of 32-element
    blocks: the zero-padded partial final block of "Scale ownership and the
    GEMM dataflow".  Zeros raise no block amax and add nothing to a block
    sum.  x itself when K is a multiple of 32."""
    rows, k = x.shape
    kp = -(-k // BLOCK) * BLOCK
    if kp == k:
        return x
    out = np.zeros((rows, kp), dtype=x.dtype)
    out[:, :k] = x
    return out


@dataclass
class MxBlocks:
    codes: np.ndarray   # uint8 [rows, K]
    scales: np.ndarray  # uint8 [rows, ceil(K/32)], E8M0 bytes, canonical order
    fmt: Fp8Format


def quantize_rows(x: np.ndarray, fmt, rule: str = "floor", rand=None) -> MxBlocks:
    """MX-quantize along the last axis (K) of a [rows, K] float64 array.

    Per 32-element block: amax = max |x|; S = 2^e from the scale rule;
    code = encode_sat_rne(x / S), or encode_sat_sr(x / S, rand) when a
    [rows, K] array of 16-bit random integers is given.  A block holding NaN
    or Inf takes scale 0xFF and NaN codes.  When K is not a multiple of 32
    the final block is the zero-padded partial block (pad_final_block); the
    codes of the padding are not returned.
    """
    f = fmt_of(fmt)
    x = np.asarray(x, dtype=np.float64)
    rows, k = x.shape
    x = pad_final_block(x)
    nb = x.shape[1] // BLOCK
    blocks = x.reshape(rows, nb, BLOCK)
    bad = ~np.all(np.isfinite(blocks), axis=2)
    amax = np.max(np.abs(np.where(np.isfinite(blocks), blocks, 0.0)), axis=2)
    if rule == "floor":
        e = scale_exponent_floor(f, amax)
    elif rule == "ceil":
        e = scale_exponent_ceil(f, amax)
    else:
        raise ValueError(rule)
    scaled = np.ldexp(blocks, -e[:, :, None])
    finite_scaled = np.where(np.isfinite(blocks), scaled, 0.0)
    if rand is None:
        codes = encode_sat_rne(f, finite_scaled)
    else:
        r = pad_final_block(np.asarray(rand, dtype=np.int64)).reshape(rows, nb, BLOCK)
        codes = encode_sat_sr(f, finite_scaled, r)
    codes = np.where(bad[:, :, None], np.uint8(f.nan_code), codes)
    scales = (e + 127).astype(np.uint8)
    scales[bad] = E8M0_NAN
    return MxBlocks(codes.reshape(rows, nb * BLOCK)[:, :k].astype(np.uint8), scales, f)


def quantize(x: np.ndarray, fmt, axis: str, rule: str = "floor", rand=None) -> MxBlocks:
    """axis 'row': blocks of 1x32 along the columns of x (x is [M, K]).
    axis 'col': blocks of 32x1 along the rows of x (x is [K, N]); the codes
    come back transposed, [N, K], so that K is contiguous -- each
    orientation is derived from the original wide data, never by moving
    codes of the other orientation."""
    x = np.asarray(x, dtype=np.float64)
    if axis == "row":
        return quantize_rows(x, fmt, rule, rand)
    if axis == "col":
        return quantize_rows(x.T, fmt, rule, None if rand is None else np.asarray(rand).T)
    raise ValueError(axis)


def dequantize(q: MxBlocks) -> np.ndarray:
    """x_hat = S * decode(code), NaN where the scale is NaN."""
    vals = pad_final_block(decode_table(q.fmt)[q.codes])
    s = e8m0_values(q.scales)
    rows, k = q.codes.shape
    nb = vals.shape[1] // BLOCK
    return (vals.reshape(rows, nb, BLOCK) * s[:, :, None]).reshape(rows, nb * BLOCK)[:, :k]


@dataclass
class IncidentTrace:
    amax: np.ndarray     # [rows, ceil(K/32)] block amax over the finite values
    scales: np.ndarray   # [rows, ceil(K/32)] the selected E8M0 bytes
    clip_count: int      # finite values whose exactly scaled magnitude exceeds the format max
    zero_count: int      # finite non-zero values that encode to a zero code
    nan_blocks: int      # blocks holding NaN or Inf (scale byte 0xFF)
    binades: dict        # floor(log2|x|) -> count, over finite non-zero values


def incident_trace(x: np.ndarray, fmt, axis: str = "row", rule: str = "floor") -> IncidentTrace:
    """The numerical fields of the incident trace that "Troubleshooting
    numerical failures" asks for, for one quantization: an input histogram
    (counts per binade), the amax of every 32-element scale group, the
    selected scale bytes, clip counts and zero counts.  A value is clipped
    when its exactly scaled magnitude lies above the format's largest finite
    value (its code is that maximum whatever the rounding), and counted as a
    zero when it is finite and non-zero but its code is +0 or -0.  Blocks
    holding NaN or Inf are counted apart and excluded from both."""
    f = fmt_of(fmt)
    q = quantize(x, f, axis, rule)
    xx = np.asarray(x, dtype=np.float64)
    if axis == "col":
        xx = xx.T
    rows, k = xx.shape
    xx = pad_final_block(xx)
    nb = xx.shape[1] // BLOCK
    blocks = xx.reshape(rows, nb, BLOCK)
    finite = np.isfinite(blocks)
    bad = ~np.all(finite, axis=2)
    vals = np.where(finite, blocks, 0.0)
    amax = np.max(np.abs(vals), axis=2)
    e = q.scales.astype(np.int64) - 127
    scaled = np.ldexp(vals, -np.where(bad, 0, e)[:, :, None])
    good = ~bad[:, :, None]
    clipped = good & (np.abs(scaled) > f.max_finite)
    decoded = pad_final_block(decode_table(f)[q.codes]).reshape(rows, nb, BLOCK)
    zeros = good & (vals != 0.0) & (decoded == 0.0)
    nz = vals[(vals != 0.0) & finite]
    _, ex = np.frexp(np.abs(nz))
    binades = {}
    for b, c in zip(*np.unique(ex - 1, return_counts=True)):
        binades[int(b)] = int(c)
    return IncidentTrace(amax, q.scales, int(clipped.sum()), int(zeros.sum()), int(bad.sum()),
                         binades)


# --------------------------------------------------------------------------
# Swizzled scale layout (tensor-core operand layout; not defined by the pages)
# --------------------------------------------------------------------------

TILE_ROWS = 128
TILE_BLOCKS = 4
TILE_BYTES = TILE_ROWS * TILE_BLOCKS


def scale_bytes(rows: int, kblocks: int) -> int:
    return -(-rows // TILE_ROWS) * TILE_ROWS * -(-kblocks // TILE_BLOCKS) * TILE_BLOCKS


def swizzle_offset(r: np.ndarray, c: np.ndarray, kblocks: int) -> np.ndarray:
    """Byte offset of scale (row r, block c).  Scales are grouped in tiles of
    128 rows x 4 blocks (512 bytes), tiles ordered row-tile-major; inside a
    tile, row r sits in 16-byte line r % 32 at 4-byte slot (r % 128) // 32,
    and the block index picks the byte within the slot."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    tiles_k = -(-kblocks // TILE_BLOCKS)
    tile = (r // TILE_ROWS) * tiles_k + c // TILE_BLOCKS
    inner = (r % 32) * 16 + ((r % TILE_ROWS) // 32) * 4 + c % TILE_BLOCKS
    return tile * TILE_BYTES + inner


def swizzle_scales(scales: np.ndarray) -> np.ndarray:
    """Canonical [rows, kblocks] scale bytes -> padded swizzled byte buffer.
    Padding bytes are 0."""
    rows, kb = scales.shape
    out = np.zeros(scale_bytes(rows, kb), dtype=np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
    out[swizzle_offset(r, c, kb)] = scales
    return out


def unswizzle_scales(buf: np.ndarray, rows: int, kblocks: int) -> np.ndarray:
    r, c = np.meshgrid(np.arange(rows), np.arange(kblocks), indexing="ij")
    return np.asarray(buf)[swizzle_offset(r, c, kblocks)]


def grouped_scale_rows(offsets) -> np.ndarray:
    """Start row of each group in the per-group padded scale layout: group g's
    scales begin at sum_{h<g} roundup(m_h, 128) rows."""
    offsets = np.asarray(offsets, dtype=np.int64)
    sizes = np.diff(offsets)
    padded = -(-sizes // TILE_ROWS) * TILE_ROWS
    return np.concatenate([[0], np.cumsum(padded)])


def grouped_scale_bytes(total_rows: int, groups: int, kblocks: int) -> int:
    """Upper bound of the per-group padded scale buffer for any split of
    total_rows into `groups` groups."""
    rows = (-(-total_rows // TILE_ROWS) + groups) * TILE_ROWS
    return scale_bytes(rows, kblocks)


def swizzle_scales_grouped(scales: np.ndarray, offsets) -> np.ndarray:
    """Rowwise scales of concatenated groups -> per-group padded swizzled
    buffer: each group is laid out as its own swizzled matrix starting at a
    128-row tile boundary.  Padding bytes are 0."""
    rows, kb = scales.shape
    offsets = np.asarray(offsets, dtype=np.int64)
    groups = len(offsets) - 1
    starts = grouped_scale_rows(offsets)
    out = np.zeros(grouped_scale_bytes(rows, groups, kb), dtype=np.uint8)
    tiles_k = -(-kb // TILE_BLOCKS)
    for g in range(groups):
        lo, hi = offsets[g], offsets[g + 1]
        if hi == lo:
            continue
        part = swizzle_scales(scales[lo:hi])
        base = starts[g] // TILE_ROWS * tiles_k * TILE_BYTES
        out[base:base + part.size] = part
    return out


# --------------------------------------------------------------------------
# Container layout of the 6- and 4-bit element codes (tensor-core operand
# layout; not defined by the pages)
# --------------------------------------------------------------------------

CONTAINER_ELEMS = 16      # elements per 16-byte container along K


def pack_container(codes: np.ndarray, fmt) -> np.ndarray:
    """One code per element [rows, K] -> the byte layout the operand takes in
    memory.  FP8 codes are their own bytes.  For 6- and 4-bit formats every
    run of 16 elements along K occupies 16 bytes: the 16 codes packed
    little-endian (element i at bits [i*w, i*w + w) of the run), followed by
    zero bytes (8 for w = 4, 4 for w = 6).  Layout only: no arithmetic on
    values.  parity unpinned on the CPU: pinned by the tensor core consuming
    bytes written by this function."""
    f = fmt_of(fmt)
    codes = np.asarray(codes, dtype=np.uint8)
    if f.bits == 8:
        return codes.copy()
    rows, k = codes.shape
    if k % CONTAINER_ELEMS:
        raise ValueError("K must be a multiple of 16")
    runs = codes.reshape(rows, k // CONTAINER_ELEMS, CONTAINER_ELEMS).astype(np.uint32)
    out = np.zeros((rows, k // CONTAINER_ELEMS, 16), dtype=np.uint32)
    for i in range(CONTAINER_ELEMS):
        off = i * f.bits
        byte, shift = off // 8, off % 8
        val = runs[:, :, i] << shift          # at most 13 bits
        out[:, :, byte] |= val & 0xFF
        if shift + f.bits > 8:
            out[:, :, byte + 1] |= val >> 8
    return out.astype(np.uint8).reshape(rows, k)


def unpack_container(buf: np.ndarray, fmt) -> np.ndarray:
    """Inverse of pack_container (padding bytes are ignored)."""
    f = fmt_of(fmt)
    buf = np.asarray(buf, dtype=np.uint8)
    if f.bits == 8:
        return buf.copy()
    rows, k = buf.shape
    b = buf.reshape(rows, k // CONTAINER_ELEMS, 16).astype(np.uint32)
    out = np.zeros((rows, k // CONTAINER_ELEMS, CONTAINER_ELEMS), dtype=np.uint32)
    mask = (1 << f.bits) - 1
    for i in range(CONTAINER_ELEMS):
        off = i * f.bits
        byte, shift = off // 8, off % 8
        val = b[:, :, byte] >> shift
        if shift + f.bits > 8:
            val |= b[:, :, byte + 1] << (8 - shift)
        out[:, :, i] = val & mask
    return out.astype(np.uint8).reshape(rows, k)


def pack_dense(codes: np.ndarray, fmt) -> np.ndarray:
    """One code per element [rows, K] -> packed storage [rows, K * w / 8]:
    the row is one little-endian bit string with element i at bits
    [i*w, i*w + w), w = 4 or 6 (two E2M1 codes per byte, four E2M3 / E3M2
    codes per three bytes) -- the payload the page counts for narrow MX
    elements, with none of the container's padding.  Layout only: no
    arithmetic on values."""
    f = fmt_of(fmt)
    codes = np.asarray(codes, dtype=np.uint8)
    if f.bits == 8:
        return codes.copy()
    rows, k = codes.shape
    if (k * f.bits) % 8:
        raise ValueError("K * w must fill whole bytes")
    out = np.zeros((rows, k * f.bits // 8), dtype=np.uint32)
    for i in range(k):
        off = i * f.bits
        byte, shift = off // 8, off % 8
        val = codes[:, i].astype(np.uint32) << shift
        out[:, byte] |= val & 0xFF
        if shift + f.bits > 8:
            out[:, byte + 1] |= val >> 8
    return out.astype(np.uint8)


def unpack_dense(buf: np.ndarray, fmt) -> np.ndarray:
    """Inverse of pack_dense."""
    f = fmt_of(fmt)
    buf = np.asarray(buf, dtype=np.uint8)
    if f.bits == 8:
        return buf.copy()
    rows, nbytes = buf.shape
    k = nbytes * 8 // f.bits
    b = buf.astype(np.uint32)
    out = np.zeros((rows, k), dtype=np.uint32)
    mask = (1 << f.bits) - 1
    for i in range(k):
        off = i * f.bits
        byte, shift = off // 8, off % 8
        val = b[:, byte] >> shift
        if shift + f.bits > 8:
            val |= b[:, byte + 1] << (8 - shift)
        out[:, i] = val & mask
    return out.astype(np.uint8)


# --------------------------------------------------------------------------
# Block-scaled GEMM
# --------------------------------------------------------------------------


def gemm(a: MxBlocks, b: MxBlocks):
    """Y[i, j] = sum_b S_A[i, b] S_B[j, b] sum_{k in b} A~[i, k] B~[j, k].

    A is [M, K] and B is [N, K] (the K-contiguous W^T), both quantized along
    K.  The inner per-block sums are a float64 matmul of decoded codes (each
    product is exact); the scale products multiply each block's partial sum
    before the outer sum, as the definition states.  A partial final block
    (K not a multiple of 32) sums its K % 32 products (zero padding adds
    nothing).  Also returns
    T[i, j] = sum_k |A_hat[i, k] B_hat[j, k]|, the magnitude the GEMM
    tolerance is relative to.
    """
    m, k = a.codes.shape
    n, k2 = b.codes.shape
    if k != k2:
        raise ValueError("K mismatch")
    av = pad_final_block(decode_table(a.fmt)[a.codes])
    bv = pad_final_block(decode_table(b.fmt)[b.codes])
    nb = av.shape[1] // BLOCK
    av = av.reshape(m, nb, BLOCK)
    bv = bv.reshape(n, nb, BLOCK)
    sa = e8m0_values(a.scales)
    sb = e8m0_values(b.scales)
    y = np.zeros((m, n), dtype=np.float64)
    t = np.zeros((m, n), dtype=np.float64)
    for blk in range(nb):
        partial = av[:, blk, :] @ bv[:, blk, :].T
        sprod = sa[:, blk][:, None] * sb[:, blk][None, :]
        y += sprod * partial
        t += sprod * (np.abs(av[:, blk, :]) @ np.abs(bv[:, blk, :]).T)
    return y, t


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + exp(-z)) in float64 (exp overflow gives -0 / 0)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


ACTIVATIONS = {"none": lambda z: np.asarray(z, dtype=np.float64), "silu": silu}


def gemm_bias_act(a: MxBlocks, b: MxBlocks, bias=None, act: str = "none"):
    """Epilogue of the kernel contract: out = act(Y + bias[None, :]) with Y the
    block-scaled GEMM; bias is one value per output column (or None).
    Returns (out, Y + bias, T)."""
    y, t = gemm(a, b)
    z = y if bias is None else y + np.asarray(bias, dtype=np.float64)[None, :]
    return ACTIVATIONS[act](z), z, t


def grouped_gemm(a: MxBlocks, offsets, b_groups):
    """Per expert g: Y[o_g:o_{g+1}] = gemm(A[o_g:o_{g+1}], B_g).  b_groups is a
    list of MxBlocks, one [N, K] operand per group."""
    offsets = np.asarray(offsets, dtype=np.int64)
    n = b_groups[0].codes.shape[0]
    m = a.codes.shape[0]
    y = np.zeros((m, n))
    t = np.zeros((m, n))
    for g in range(len(offsets) - 1):
        lo, hi = offsets[g], offsets[g + 1]
        if hi == lo:
            continue
        sub = MxBlocks(a.codes[lo:hi], a.scales[lo:hi], a.fmt)
        y[lo:hi], t[lo:hi] = gemm(sub, b_groups[g])
    return y, t


def quantize_grouped_cols(x: np.ndarray, offsets, fmt, rule: str = "floor"):
    """Columnwise MX quantization inside each group of rows of a [total, C]
    array (the token-major activations or output gradients of a mixture of
    experts).  Group g is X_g = x[o_g:o_{g+1}]; its 32-row blocks start at
    the group's first row, so no block spans two groups, and a final
    partial block is completed with zero rows (the page's zero-padded final
    block).  Zeros raise no amax and add nothing to a sum.  Returns one
    MxBlocks per group: codes [C, roundup(m_g, 32)], K = the group's tokens.
    """
    x = np.asarray(x, dtype=np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    out = []
    for g in range(len(offsets) - 1):
        lo, hi = int(offsets[g]), int(offsets[g + 1])
        padded = np.zeros((-(-(hi - lo) // BLOCK) * BLOCK, x.shape[1]))
        padded[:hi - lo] = x[lo:hi]
        out.append(quantize(padded, fmt, "col", rule))
    return out


def grouped_wgrad(a_groups, b_groups):
    """Per expert g: Y[g] = gemm(A_g, B_g), where A_g [M, K_g] and B_g [N, K_g]
    are columnwise quantizations over that expert's tokens (K_g its padded
    token count): the weight gradient of each expert, contracted over the
    expert's own tokens only.  An expert without tokens gets Y[g] = 0.
    Returns (Y [G, M, N], T [G, M, N])."""
    groups = len(a_groups)
    m = a_groups[0].codes.shape[0]
    n = b_groups[0].codes.shape[0]
    y = np.zeros((groups, m, n))
    t = np.zeros((groups, m, n))
    for g in range(groups):
        if a_groups[g].codes.shape[1]:
            y[g], t[g] = gemm(a_groups[g], b_groups[g])
    return y, t


def pack_grouped_cols(groups_mx, offsets, ldq: int):
    """Side-by-side layout of per-group columnwise operands along K: group
    g's codes occupy columns [s_g, s_g + roundup(m_g, 32)) of a [C, ldq]
    matrix, s_g = sum_{h<g} roundup(m_h, 128) (every group starts at a
    128-column boundary, the start of a scale tile); the rest of the group's
    128-column segment holds code 0 and scale byte 0.  Returns (codes
    [C, ldq], canonical scales [C, ldq / 32]).  Layout only: no arithmetic."""
    starts = grouped_scale_rows(offsets)
    c = groups_mx[0].codes.shape[0]
    if starts[-1] > ldq or ldq % TILE_ROWS:
        raise ValueError("ldq too small or not a multiple of 128")
    codes = np.zeros((c, ldq), dtype=np.uint8)
    scales = np.zeros((c, ldq // BLOCK), dtype=np.uint8)
    for g, q in enumerate(groups_mx):
        s0 = int(starts[g])
        kp = q.codes.shape[1]
        codes[:, s0:s0 + kp] = q.codes
        scales[:, s0 // BLOCK:(s0 + kp) // BLOCK] = q.scales
    return codes, scales


# --------------------------------------------------------------------------
# Helpers used by the pins and the parity tests
# --------------------------------------------------------------------------


def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return u32.view(np.float32).astype(np.float64)


def exact_gemm_fraction(a: MxBlocks, b: MxBlocks):
    """Exact rational Y for tiny shapes (Python Fractions), for pins."""
    m, k = a.codes.shape
    n = b.codes.shape[0]
    ta = [Fraction(v) if np.isfinite(v) else None for v in decode_table(a.fmt)]
    tb = [Fraction(v) if np.isfinite(v) else None for v in decode_table(b.fmt)]
    out = [[Fraction(0)] * n for _ in range(m)]
    for i in range(m):
        for j in range(n):
            acc = Fraction(0)
            for blk in range(-(-k // BLOCK)):
                sa = Fraction(2) ** (int(a.scales[i, blk]) - 127)
                sb = Fraction(2) ** (int(b.scales[j, blk]) - 127)
                part = sum(ta[a.codes[i, kk]] * tb[b.codes[j, kk]]
                           for kk in range(blk * BLOCK, min(k, (blk + 1) * BLOCK)))
                acc += sa * sb * part
            out[i][j] = acc
    return out
