"""Shared helpers of the parity tests: oracle calls on torch inputs and the
GEMM acceptance bound.  Test infrastructure; imports the oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

from oracle import mx_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# GEMM acceptance (FP32 accumulation): |y - y_ref| <= REL_TOL * T, where
# T = sum_k |a_hat * b_hat|; BF16 outputs may additionally be one BF16 ulp
# of y_ref off (round-to-nearest-even of the FP32 result).
REL_TOL = 1e-4


def ensure_built():
    lib = os.path.join(ROOT, "mxfp8_block_scaled_mx_gb300", "libmx.so")
    if not os.path.exists(lib):
        from mxfp8_block_scaled_mx_gb300 import build
        build.build()
    return lib


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 / fp32 tensor."""
    return t.detach().to("cpu").float().double().numpy()


def oracle_quant(x_bf16: torch.Tensor, fmt: str, axis: str, rule: str = "floor"):
    """Oracle quantization of a bf16 tensor; returns (MxBlocks, swizzled scales)."""
    q = O.quantize(to_f64(x_bf16), fmt, axis, rule)
    return q, O.swizzle_scales(q.scales)


def mx_from_oracle(q: O.MxBlocks, device="cuda"):
    """Oracle codes and swizzled scales as device tensors for the GEMM."""
    from mxfp8_block_scaled_mx_gb300 import MxTensor
    codes = torch.from_numpy(np.ascontiguousarray(q.codes)).to(device)
    scales = torch.from_numpy(O.swizzle_scales(q.scales)).to(device)
    return MxTensor(codes, scales, q.fmt.name)


def canonical_scales(gpu_scales: torch.Tensor, rows: int, k: int) -> np.ndarray:
    return O.unswizzle_scales(gpu_scales.cpu().numpy(), rows, k // 32)


def bf16_ulp(y: np.ndarray) -> np.ndarray:
    a = np.abs(y)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


# Incident-trace counts read off GPU-quantized tensors (test id, what,
# values, clipped, zeroed, NaN/Inf blocks); conftest prints them.
INCIDENT_LOG: list = []


def incident_counts(x_bf16: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, fmt: str,
                    axis: str):
    """Clip and zero counts of a quantization read off its codes and
    swizzled scales (the incident trace's definitions: a finite value is
    clipped when its value over the block scale exceeds the format max, and
    zeroed when it is non-zero and its code decodes to zero)."""
    f = O.fmt_of(fmt)
    x = to_f64(x_bf16)
    if axis == "col":
        x = x.T
    rows, k = x.shape
    sc = O.unswizzle_scales(scales.cpu().numpy(), rows, k // 32)
    blocks = x.reshape(rows, k // 32, 32)
    bad = (sc == O.E8M0_NAN)
    good = ~bad[:, :, None] & np.isfinite(blocks)
    e = sc.astype(np.int64) - 127
    scaled = np.ldexp(np.where(good, blocks, 0.0), -np.where(bad, 0, e)[:, :, None])
    dec = O.decode_table(f)[codes.cpu().numpy().reshape(rows, k // 32, 32)]
    clipped = int((good & (np.abs(scaled) > f.max_finite)).sum())
    zeroed = int((good & (blocks != 0.0) & (dec == 0.0)).sum())
    return clipped, zeroed, int(bad.sum())


# Observed GEMM accuracy, one record per checked block of outputs:
# (test id, output dtype, max error / allowed bound, max |y - y_ref| / T over
# entries with T > 0, entries checked).  conftest prints a summary.
ERROR_LOG: list = []


def gemm_error_ratio(y_gpu: torch.Tensor, y_ref: np.ndarray, t_ref: np.ndarray,
                     out_dtype: str) -> float:
    """max |y - y_ref| / allowed over all entries (<= 1 passes)."""
    y = to_f64(y_gpu)
    allowed = REL_TOL * t_ref
    if out_dtype == "bf16":
        allowed = allowed + bf16_ulp(y_ref)
    allowed = np.maximum(allowed, 1e-300)
    err = np.abs(y - y_ref)
    assert np.isfinite(y).all(), "non-finite GEMM output"
    ratio = float((err / allowed).max()) if err.size else 0.0
    pos = t_ref > 0
    rel_t = float((err[pos] / t_ref[pos]).max()) if pos.any() else 0.0
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    ERROR_LOG.append((test, out_dtype, ratio, rel_t, int(err.size)))
    return ratio


def assert_gemm_close(y_gpu, y_ref, t_ref, out_dtype):
    r = gemm_error_ratio(y_gpu, y_ref, t_ref, out_dtype)
    assert r <= 1.0, f"GEMM error {r:.3g} x the allowed bound"
    return r
