"""MXFP8 training matmul for GB300: a thin Python binding over libmx.so.

The binding only marshals arguments: every step of quantization and of the
block-scaled GEMM runs in the CUDA kernels behind the C ABI declared in
include/mx.h.  PyTorch supplies device memory and the current stream.
There is no CPU fallback: calling any entry point without the built
library raises.

Low-level functions carry the C names (mx_quantize, mx_quantize_grouped,
mx_gemm, mx_grouped_gemm, mx_device_status, ...) and take raw pointers;
`quantize`, `quantize_grouped`, `gemm` and `grouped_gemm` wrap them for
torch tensors.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmx.so")

MX_OK = 0
STATUS_NAMES = {0: "MX_OK", 1: "MX_ERR_INVALID_ARG", 2: "MX_ERR_MISALIGNED",
                3: "MX_ERR_UNSUPPORTED", 4: "MX_ERR_CUDA", 5: "MX_ERR_TIMEOUT",
                6: "MX_ERR_DEVICE_ARG"}
FMT = {"e4m3": 0, "e5m2": 1, "e2m3": 2, "e3m2": 3, "e2m1": 4,
       "e2m3_packed": 5, "e3m2_packed": 6, "e2m1_packed": 7}
# bits of storage per element: 8 for FP8 and the container layout of the
# narrow formats, the code width for packed storage
STORAGE_BITS = {"e2m3_packed": 6, "e3m2_packed": 6, "e2m1_packed": 4}


def storage_bytes(fmt: str, elems: int) -> int:
    """Bytes that `elems` consecutive codes of `fmt` occupy along K."""
    return elems * STORAGE_BITS.get(fmt, 8) // 8


def storage_elems(fmt: str, nbytes: int) -> int:
    """Codes of `fmt` held by `nbytes` bytes along K."""
    return nbytes * 8 // STORAGE_BITS.get(fmt, 8)


DTYPE = {"bf16": 0, "fp32": 1}
_X_DTYPE = {torch.bfloat16: DTYPE["bf16"], torch.float32: DTYPE["fp32"]}  # quantizer inputs
AXIS = {"row": 1, "col": 2, "both": 3}
RULE = {"floor": 0, "ceil": 1}

ACT = {"none": 0, "silu": 1}

EXPORTS = ("mx_scale_bytes", "mx_grouped_scale_bytes", "mx_grouped_cols_capacity",
           "mx_quantize", "mx_quantize_sr", "mx_quantize_grouped", "mx_quantize_grouped_ex",
           "mx_gemm", "mx_gemm_bias_act", "mx_grouped_gemm", "mx_grouped_gemm_bcat",
           "mx_grouped_gemm_wgrad", "mx_device_status", "mx_status_str",
           "mx_set_wait_timeout_ns", "mx_selftest_wait_timeout")


class MxError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def _declare(lib):
    c = ctypes
    i64, i32, u64, vp = c.c_int64, c.c_int32, c.c_uint64, c.c_void_p
    lib.mx_scale_bytes.argtypes = [i64, i64]
    lib.mx_scale_bytes.restype = c.c_size_t
    lib.mx_grouped_scale_bytes.argtypes = [i64, i32, i64]
    lib.mx_grouped_scale_bytes.restype = c.c_size_t
    lib.mx_quantize.argtypes = [vp, c.c_int, i64, i64, i64, c.c_int, c.c_int, c.c_int,
                                vp, vp, vp, vp, vp]
    lib.mx_quantize.restype = c.c_int
    lib.mx_quantize_sr.argtypes = [vp, c.c_int, i64, i64, i64, vp, i64, c.c_int, c.c_int,
                                   c.c_int, vp, vp, vp, vp, vp]
    lib.mx_quantize_sr.restype = c.c_int
    lib.mx_quantize_grouped.argtypes = [vp, c.c_int, i64, i64, i64, c.c_int, c.c_int, i32, vp,
                                        vp, vp, vp]
    lib.mx_quantize_grouped.restype = c.c_int
    lib.mx_grouped_cols_capacity.argtypes = [i64, i32]
    lib.mx_grouped_cols_capacity.restype = i64
    lib.mx_quantize_grouped_ex.argtypes = [vp, c.c_int, i64, i64, i64, c.c_int, c.c_int, c.c_int,
                                           i32, vp, vp, vp, vp, i64, vp, vp]
    lib.mx_quantize_grouped_ex.restype = c.c_int
    lib.mx_grouped_gemm_bcat.argtypes = [i32, vp, i64, i64, i64, vp, vp, c.c_int, vp, i64, vp,
                                         c.c_int, vp, c.c_int, vp]
    lib.mx_grouped_gemm_bcat.restype = c.c_int
    lib.mx_grouped_gemm_wgrad.argtypes = [i32, vp, i64, i64, i64, i64, vp, vp, c.c_int, vp, vp,
                                          c.c_int, vp, c.c_int, vp]
    lib.mx_grouped_gemm_wgrad.restype = c.c_int
    lib.mx_gemm.argtypes = [i64, i64, i64, vp, vp, c.c_int, vp, vp, c.c_int, vp, c.c_int, i64, vp]
    lib.mx_gemm.restype = c.c_int
    lib.mx_gemm_bias_act.argtypes = [i64, i64, i64, vp, vp, c.c_int, vp, vp, c.c_int, vp, c.c_int,
                                     vp, c.c_int, i64, vp]
    lib.mx_gemm_bias_act.restype = c.c_int
    lib.mx_grouped_gemm.argtypes = [i32, vp, i64, i64, i64, vp, vp, c.c_int, vp, vp, c.c_int, vp,
                                    c.c_int, vp]
    lib.mx_grouped_gemm.restype = c.c_int
    lib.mx_device_status.argtypes = [vp]
    lib.mx_device_status.restype = c.c_int
    lib.mx_status_str.argtypes = [c.c_int]
    lib.mx_status_str.restype = c.c_char_p
    lib.mx_set_wait_timeout_ns.argtypes = [u64]
    lib.mx_set_wait_timeout_ns.restype = c.c_int
    lib.mx_selftest_wait_timeout.argtypes = [u64, vp]
    lib.mx_selftest_wait_timeout.restype = c.c_int


def lib():
    """The loaded libmx.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m mxfp8_block_scaled_mx_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        _declare(handle)
        _lib = handle
    return _lib


def _check(fn: str, status: int):
    if status != MX_OK:
        raise MxError(fn, status)


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


# The C ABI takes raw pointers and cannot see buffer sizes: the tensor API
# checks them before every call, so that no kernel reads or writes past a
# caller's tensor.  Every tensor must also live on the current CUDA device
# (the device whose stream the call is enqueued on); the C ABI refuses
# other devices' memory too.

def _on_current_device(t: torch.Tensor, what: str):
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor, got {t.device}")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{what} must be on the current CUDA device "
                         f"(cuda:{torch.cuda.current_device()}), got {t.device}")


def _require_codes(t: torch.Tensor, shape, what: str):
    _on_current_device(t, what)
    if (t.dtype != torch.uint8 or not t.is_cuda or tuple(t.shape) != tuple(shape)
            or not t.is_contiguous()):
        raise ValueError(f"{what}: codes must be a contiguous CUDA uint8 tensor of shape "
                         f"{tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


def _require_scales(t: torch.Tensor, nbytes: int, what: str):
    _on_current_device(t, what)
    if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous() or t.numel() < nbytes:
        raise ValueError(f"{what}: scales must be a contiguous CUDA uint8 tensor of at least "
                         f"{nbytes} bytes, got {t.numel()}")


def _require_out(out: torch.Tensor, shape, dtype, contiguous: bool):
    _on_current_device(out, "out")
    if out.dtype != dtype or not out.is_cuda or tuple(out.shape) != tuple(shape):
        raise ValueError(f"out must be a CUDA {dtype} tensor of shape {tuple(shape)}, got "
                         f"{out.dtype} {tuple(out.shape)}")
    if out.stride(-1) != 1 or (contiguous and not out.is_contiguous()):
        raise ValueError("out must have unit column stride" +
                         (" and be contiguous" if contiguous else ""))


def _require_offsets(offsets: torch.Tensor) -> int:
    _on_current_device(offsets, "offsets")
    if offsets.dtype != torch.int32 or not offsets.is_cuda or offsets.dim() != 1 or \
            not offsets.is_contiguous() or offsets.numel() < 2:
        raise ValueError("offsets must be a contiguous 1-D CUDA int32 tensor of groups + 1 entries")
    return offsets.numel() - 1


# ---------------------------------------------------------------- C-named calls

def mx_scale_bytes(rows: int, k: int) -> int:
    return int(lib().mx_scale_bytes(rows, k))


def mx_grouped_scale_bytes(total_rows: int, groups: int, k: int) -> int:
    return int(lib().mx_grouped_scale_bytes(total_rows, groups, k))


def mx_quantize(x, x_dtype, rows, cols, ldx, fmt, axis, rule, q_row, s_row, q_col, s_col,
                stream) -> int:
    return lib().mx_quantize(x, x_dtype, rows, cols, ldx, fmt, axis, rule, q_row, s_row, q_col,
                             s_col, stream)


def mx_quantize_sr(x, x_dtype, rows, cols, ldx, rbits, ldr, fmt, axis, rule, q_row, s_row, q_col,
                   s_col, stream) -> int:
    return lib().mx_quantize_sr(x, x_dtype, rows, cols, ldx, rbits, ldr, fmt, axis, rule, q_row,
                                s_row, q_col, s_col, stream)


def mx_quantize_grouped(x, x_dtype, total_rows, cols, ldx, fmt, rule, groups, d_offsets, q, s,
                        stream) -> int:
    return lib().mx_quantize_grouped(x, x_dtype, total_rows, cols, ldx, fmt, rule, groups,
                                     d_offsets, q, s, stream)


def mx_grouped_cols_capacity(total_rows: int, groups: int) -> int:
    return int(lib().mx_grouped_cols_capacity(total_rows, groups))


def mx_quantize_grouped_ex(x, x_dtype, total_rows, cols, ldx, fmt, axis, rule, groups, d_offsets,
                           q_row, s_row, q_col, ldq_col, s_col, stream) -> int:
    return lib().mx_quantize_grouped_ex(x, x_dtype, total_rows, cols, ldx, fmt, axis, rule,
                                        groups, d_offsets, q_row, s_row, q_col, ldq_col, s_col,
                                        stream)


def mx_grouped_gemm_bcat(groups, d_offsets, total_m, n, k, a, sa, fa, b, ldb, sb, fb, y, y_dtype,
                         stream) -> int:
    return lib().mx_grouped_gemm_bcat(groups, d_offsets, total_m, n, k, a, sa, fa, b, ldb, sb, fb,
                                      y, y_dtype, stream)


def mx_grouped_gemm_wgrad(groups, d_offsets, total_tokens, m, n, ldk, a, sa, fa, b, sb, fb, y,
                          y_dtype, stream) -> int:
    return lib().mx_grouped_gemm_wgrad(groups, d_offsets, total_tokens, m, n, ldk, a, sa, fa, b,
                                       sb, fb, y, y_dtype, stream)


def mx_gemm(m, n, k, a, sa, fa, b, sb, fb, y, y_dtype, ldy, stream) -> int:
    return lib().mx_gemm(m, n, k, a, sa, fa, b, sb, fb, y, y_dtype, ldy, stream)


def mx_gemm_bias_act(m, n, k, a, sa, fa, b, sb, fb, bias, act, y, y_dtype, ldy, stream) -> int:
    return lib().mx_gemm_bias_act(m, n, k, a, sa, fa, b, sb, fb, bias, act, y, y_dtype, ldy,
                                  stream)


def mx_grouped_gemm(groups, d_offsets, total_m, n, k, a, sa, fa, b, sb, fb, y, y_dtype,
                    stream) -> int:
    return lib().mx_grouped_gemm(groups, d_offsets, total_m, n, k, a, sa, fa, b, sb, fb, y,
                                 y_dtype, stream)


def mx_device_status(stream=None) -> int:
    return lib().mx_device_status(_stream(stream))


def mx_status_str(status: int) -> str:
    return lib().mx_status_str(status).decode()


def mx_set_wait_timeout_ns(ns: int) -> int:
    return lib().mx_set_wait_timeout_ns(ns)


def mx_selftest_wait_timeout(ns: int, stream=None) -> int:
    return lib().mx_selftest_wait_timeout(ns, _stream(stream))


# ---------------------------------------------------------------- tensor API

@dataclass
class MxTensor:
    """MX operand: codes [rows, k] (K contiguous) and swizzled E8M0 scales."""
    codes: torch.Tensor
    scales: torch.Tensor
    fmt: str

    @property
    def rows(self) -> int:
        return self.codes.shape[-2]

    @property
    def k(self) -> int:
        """Elements along K (packed storage holds fewer bytes than elements)."""
        return storage_elems(self.fmt, self.codes.shape[-1])


def quantize(x: torch.Tensor, fmt: str = "e4m3", axis: str = "row", rule: str = "floor",
             stream=None, rand: torch.Tensor | None = None):
    """bf16 or fp32 [rows, cols] -> MxTensor (axis 'row' or 'col') or a
    (row, col) pair (axis 'both').  Column-wise codes come back as [cols,
    rows].  With `rand` (16-bit random integers, int16 [rows, cols]) the
    codes use stochastic rounding."""
    if x.dtype not in _X_DTYPE or x.dim() != 2 or not x.is_cuda:
        raise ValueError("x must be a 2-D bf16 or fp32 CUDA tensor")
    _on_current_device(x, "x")
    if x.stride(1) != 1:
        raise ValueError("x must be row-major with unit column stride")
    rows, cols = x.shape
    dev = x.device
    q_row = s_row = q_col = s_col = None
    if axis in ("row", "both"):
        q_row = torch.empty((rows, storage_bytes(fmt, cols)), dtype=torch.uint8, device=dev)
        s_row = torch.empty(max(mx_scale_bytes(rows, cols), 1), dtype=torch.uint8, device=dev)
    if axis in ("col", "both"):
        q_col = torch.empty((cols, storage_bytes(fmt, rows)), dtype=torch.uint8, device=dev)
        s_col = torch.empty(max(mx_scale_bytes(cols, rows), 1), dtype=torch.uint8, device=dev)
    if rand is None:
        st = mx_quantize(_ptr(x), _X_DTYPE[x.dtype], rows, cols, x.stride(0), FMT[fmt], AXIS[axis],
                         RULE[rule], _ptr(q_row), _ptr(s_row), _ptr(q_col), _ptr(s_col),
                         _stream(stream))
        _check("mx_quantize", st)
    else:
        if rand.dtype != torch.int16 or rand.shape != x.shape or not rand.is_cuda:
            raise ValueError("rand must be a CUDA int16 tensor shaped like x")
        _on_current_device(rand, "rand")
        if rand.stride(1) != 1:
            raise ValueError("rand must have unit column stride")
        st = mx_quantize_sr(_ptr(x), _X_DTYPE[x.dtype], rows, cols, x.stride(0), _ptr(rand),
                            rand.stride(0), FMT[fmt], AXIS[axis], RULE[rule], _ptr(q_row),
                            _ptr(s_row), _ptr(q_col), _ptr(s_col), _stream(stream))
        _check("mx_quantize_sr", st)
    row = MxTensor(q_row, s_row, fmt) if q_row is not None else None
    col = MxTensor(q_col, s_col, fmt) if q_col is not None else None
    if axis == "row":
        return row
    if axis == "col":
        return col
    return row, col


def quantize_grouped(x: torch.Tensor, offsets: torch.Tensor, fmt: str = "e4m3",
                     rule: str = "floor", stream=None, axis: str = "row", ldq: int | None = None):
    """MX quantization of expert-grouped tokens x[total, cols]; offsets is a
    device int32 tensor of groups+1 entries.
    axis 'row': MxTensor [total, cols] with the per-group padded scale layout
    that grouped_gemm reads.  axis 'col': MxTensor [cols, ldq] holding every
    group's columnwise codes in its own 128-padded token segment (blocks
    start at the group's first token; the final partial block is
    zero-padded), the operand layout of grouped_gemm_wgrad; ldq defaults to
    mx_grouped_cols_capacity(total, groups).  axis 'both': (row, col) from
    one read."""
    if x.dtype not in _X_DTYPE or x.dim() != 2 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("x must be a row-major 2-D bf16 or fp32 CUDA tensor")
    _on_current_device(x, "x")
    groups = _require_offsets(offsets)
    rows, cols = x.shape
    q_row = s_row = q_col = s_col = None
    if axis in ("row", "both"):
        q_row = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
        s_row = torch.zeros(max(mx_grouped_scale_bytes(rows, groups, cols), 1), dtype=torch.uint8,
                            device=x.device)
    if axis in ("col", "both"):
        if ldq is None:
            ldq = mx_grouped_cols_capacity(rows, groups)
        q_col = torch.zeros((cols, ldq), dtype=torch.uint8, device=x.device)
        s_col = torch.zeros(max(mx_scale_bytes(cols, ldq), 1), dtype=torch.uint8, device=x.device)
    if axis == "row":
        st = mx_quantize_grouped(_ptr(x), _X_DTYPE[x.dtype], rows, cols, x.stride(0), FMT[fmt],
                                 RULE[rule], groups, _ptr(offsets), _ptr(q_row), _ptr(s_row),
                                 _stream(stream))
        _check("mx_quantize_grouped", st)
        return MxTensor(q_row, s_row, fmt)
    st = mx_quantize_grouped_ex(_ptr(x), _X_DTYPE[x.dtype], rows, cols, x.stride(0), FMT[fmt],
                                AXIS[axis], RULE[rule], groups, _ptr(offsets), _ptr(q_row),
                                _ptr(s_row), _ptr(q_col), ldq or 0, _ptr(s_col), _stream(stream))
    _check("mx_quantize_grouped_ex", st)
    col = MxTensor(q_col, s_col, fmt)
    return col if axis == "col" else (MxTensor(q_row, s_row, fmt), col)


def gemm(a: MxTensor, b: MxTensor, out_dtype: str = "bf16", out: torch.Tensor | None = None,
         stream=None, bias: torch.Tensor | None = None, act: str = "none") -> torch.Tensor:
    """y[m, n] = block-scaled A[m, k] * B[n, k]^T; with `bias` (FP32 [n]) or
    `act` ("silu") the fused epilogue computes act(y + bias)."""
    m, k = a.codes.shape[0], a.k
    n, k2 = b.codes.shape[0], b.k
    if k != k2:
        raise ValueError("K mismatch")
    _require_codes(a.codes, (m, storage_bytes(a.fmt, k)), "a")
    _require_codes(b.codes, (n, storage_bytes(b.fmt, k)), "b")
    _require_scales(a.scales, mx_scale_bytes(m, k), "a")
    _require_scales(b.scales, mx_scale_bytes(n, k), "b")
    tdtype = torch.float32 if out_dtype == "fp32" else torch.bfloat16
    if out is None:
        out = torch.empty((m, n), dtype=tdtype, device=a.codes.device)
    _require_out(out, (m, n), tdtype, contiguous=False)
    if bias is None and act == "none":
        st = mx_gemm(m, n, k, _ptr(a.codes), _ptr(a.scales), FMT[a.fmt], _ptr(b.codes),
                     _ptr(b.scales), FMT[b.fmt], _ptr(out), DTYPE[out_dtype], out.stride(0),
                     _stream(stream))
        _check("mx_gemm", st)
        return out
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != n or not bias.is_cuda):
        raise ValueError("bias must be a CUDA float32 tensor of n elements")
    if bias is not None:
        _on_current_device(bias, "bias")
    st = mx_gemm_bias_act(m, n, k, _ptr(a.codes), _ptr(a.scales), FMT[a.fmt], _ptr(b.codes),
                          _ptr(b.scales), FMT[b.fmt], _ptr(bias), ACT[act], _ptr(out),
                          DTYPE[out_dtype], out.stride(0), _stream(stream))
    _check("mx_gemm_bias_act", st)
    return out


def grouped_gemm(a: MxTensor, offsets: torch.Tensor, b: MxTensor, out_dtype: str = "bf16",
                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per group g: y[o_g:o_{g+1}] = A[o_g:o_{g+1}] * B_g^T.  b.codes is
    [groups, n, k]; b.scales holds groups consecutive swizzled matrices."""
    total_m, k = a.codes.shape[0], a.k
    groups, n, k2 = b.codes.shape[0], b.codes.shape[1], b.k
    if k != k2 or _require_offsets(offsets) != groups:
        raise ValueError("shape mismatch")
    _require_codes(a.codes, (total_m, storage_bytes(a.fmt, k)), "a")
    _require_codes(b.codes, (groups, n, storage_bytes(b.fmt, k)), "b")
    _require_scales(a.scales, mx_grouped_scale_bytes(total_m, groups, k), "a")
    _require_scales(b.scales, groups * mx_scale_bytes(n, k), "b")
    tdtype = torch.float32 if out_dtype == "fp32" else torch.bfloat16
    if out is None:
        out = torch.empty((total_m, n), dtype=tdtype, device=a.codes.device)
    _require_out(out, (total_m, n), tdtype, contiguous=True)
    st = mx_grouped_gemm(groups, _ptr(offsets), total_m, n, k, _ptr(a.codes), _ptr(a.scales),
                         FMT[a.fmt], _ptr(b.codes), _ptr(b.scales), FMT[b.fmt], _ptr(out),
                         DTYPE[out_dtype], _stream(stream))
    _check("mx_grouped_gemm", st)
    return out


def grouped_gemm_bcat(a: MxTensor, offsets: torch.Tensor, b: MxTensor, out_dtype: str = "bf16",
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per group g: y[o_g:o_{g+1}] = A[o_g:o_{g+1}] * B_g^T with B_g the
    columns [g*k, (g+1)*k) of one [n, groups*k] operand (b from quantize(...,
    axis="col") of the stacked [groups*k, n] expert weights); k = a's K."""
    total_m, k = a.codes.shape[0], a.k
    n, ldb = b.codes.shape[0], b.k
    groups = _require_offsets(offsets)
    _require_codes(a.codes, (total_m, storage_bytes(a.fmt, k)), "a")
    _require_codes(b.codes, (n, storage_bytes(b.fmt, ldb)), "b")
    _require_scales(a.scales, mx_grouped_scale_bytes(total_m, groups, k), "a")
    _require_scales(b.scales, mx_scale_bytes(n, ldb), "b")
    tdtype = torch.float32 if out_dtype == "fp32" else torch.bfloat16
    if out is None:
        out = torch.empty((total_m, n), dtype=tdtype, device=a.codes.device)
    _require_out(out, (total_m, n), tdtype, contiguous=True)
    st = mx_grouped_gemm_bcat(groups, _ptr(offsets), total_m, n, k, _ptr(a.codes),
                              _ptr(a.scales), FMT[a.fmt], _ptr(b.codes), ldb, _ptr(b.scales),
                              FMT[b.fmt], _ptr(out), DTYPE[out_dtype], _stream(stream))
    _check("mx_grouped_gemm_bcat", st)
    return out


def grouped_gemm_wgrad(a: MxTensor, offsets: torch.Tensor, b: MxTensor, total_tokens: int,
                       out_dtype: str = "fp32", out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Per group g: y[g] = A_g * B_g^T over the group's tokens, with a and b
    from quantize_grouped(..., axis="col") (same offsets and ldq).  Returns
    [groups, m, n]; an expert without tokens gets zeros."""
    m, ldk = a.codes.shape[0], a.k
    n, ldk2 = b.codes.shape[0], b.k
    groups = _require_offsets(offsets)
    if ldk != ldk2:
        raise ValueError("A and B must share the token layout (ldq)")
    _require_codes(a.codes, (m, storage_bytes(a.fmt, ldk)), "a")
    _require_codes(b.codes, (n, storage_bytes(b.fmt, ldk)), "b")
    _require_scales(a.scales, mx_scale_bytes(m, ldk), "a")
    _require_scales(b.scales, mx_scale_bytes(n, ldk), "b")
    tdtype = torch.float32 if out_dtype == "fp32" else torch.bfloat16
    if out is None:
        out = torch.empty((groups, m, n), dtype=tdtype, device=a.codes.device)
    _require_out(out, (groups, m, n), tdtype, contiguous=True)
    st = mx_grouped_gemm_wgrad(groups, _ptr(offsets), total_tokens, m, n, ldk, _ptr(a.codes),
                               _ptr(a.scales), FMT[a.fmt], _ptr(b.codes), _ptr(b.scales),
                               FMT[b.fmt], _ptr(out), DTYPE[out_dtype], _stream(stream))
    _check("mx_grouped_gemm_wgrad", st)
    return out


def device_status(stream=None) -> int:
    """Synchronize and return (and clear) the device status word."""
    return mx_device_status(stream)
