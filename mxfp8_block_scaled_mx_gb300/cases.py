"""Run one hot-path kernel on one shape a few times (for profilers).

    python -m mxfp8_block_scaled_mx_gb300.cases gemm --m 4096 --n 18432 --k 7168 [--reps 3] [--fused]
    python -m mxfp8_block_scaled_mx_gb300.cases quantize --rows 16384 --cols 8192 --axis row [--sr] [--fp32] [--flush write]
    python -m mxfp8_block_scaled_mx_gb300.cases moe_quantize --tokens 65536 --experts 64 --axis col
    python -m mxfp8_block_scaled_mx_gb300.cases grouped --tokens 16384 --experts 16
    python -m mxfp8_block_scaled_mx_gb300.cases moe_dgrad --tokens 16384 --experts 16
    python -m mxfp8_block_scaled_mx_gb300.cases moe_wgrad --tokens 16384 --experts 16

Inputs are the seeded synthetic workloads; each case launches the kernel
`--reps` times after building its inputs and prints the mean event time.
"""
from __future__ import annotations

import argparse
import sys

import torch

import mxfp8_block_scaled_mx_gb300 as mx
from mxfp8_block_scaled_mx_gb300 import workloads as W


def _time(fn, reps, pre=None):
    fn()  # warm-up launch (module load, attributes)
    torch.cuda.synchronize()
    if pre is None:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps
    # one launch at a time behind `pre` (an L2 flush), timed on its own
    ts = []
    for _ in range(reps):
        pre()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ts) / reps


def _flush(kind, dev):
    """The L2 state before each timed launch: `write` adds 1 to a 256 MB
    buffer (L2 left full of dirty lines, as the bench's flush leaves it),
    `read` does that and then sums another 256 MB buffer (L2 left full of
    clean lines), `none` launches back to back."""
    if kind == "none":
        return None
    scrub = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    if kind == "write":
        return lambda: scrub.add_(1)
    clean = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    return lambda: (scrub.add_(1), clean.sum())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["gemm", "quantize", "grouped", "moe_dgrad", "moe_wgrad",
                                     "moe_quantize"])
    ap.add_argument("--m", type=int, default=4096)
    ap.add_argument("--n", type=int, default=18432)
    ap.add_argument("--k", type=int, default=7168)
    ap.add_argument("--rows", type=int, default=16384)
    ap.add_argument("--cols", type=int, default=8192)
    ap.add_argument("--axis", default="row", choices=["row", "col", "both"])
    ap.add_argument("--tokens", type=int, default=16384)
    ap.add_argument("--experts", type=int, default=16)
    ap.add_argument("--out", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--fused", action="store_true", help="gemm: FP32 bias + SiLU epilogue")
    ap.add_argument("--sr", action="store_true", help="quantize: stochastic rounding (E5M2)")
    ap.add_argument("--fp32", action="store_true", help="quantize: FP32 input (same values)")
    ap.add_argument("--flush", default="none", choices=["none", "write", "read"],
                    help="quantize: L2 state before each launch (see _flush)")
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    if a.case == "gemm":
        x, w = W.dense_forward(a.m, a.n, a.k, device=dev)
        qa = mx.quantize(x, "e4m3", "row")
        qb = mx.quantize(w, "e4m3", "col")
        del x, w
        y = torch.empty((a.m, a.n), dtype=torch.bfloat16 if a.out == "bf16" else torch.float32,
                        device=dev)
        if a.fused:  # FP32 bias + SiLU epilogue
            bias = torch.randn(a.n, generator=torch.Generator().manual_seed(3)).to(dev)
            ms = _time(lambda: mx.gemm(qa, qb, a.out, out=y, bias=bias, act="silu"), a.reps)
        else:
            ms = _time(lambda: mx.gemm(qa, qb, a.out, out=y), a.reps)
        print(f"gemm {a.m}x{a.n}x{a.k}{' bias+silu' if a.fused else ''}: {ms:.4f} ms, "
              f"{2 * a.m * a.n * a.k / ms / 1e9:.1f} TFLOP/s")
    elif a.case == "quantize":
        x = W.quantize_sweep((a.rows, a.cols), seed=1, device=dev)
        bpe = 4.0625 if a.axis == "both" else 3.03125
        if a.fp32:
            x = x.float()
            bpe += 2.0
        if a.sr:  # stochastic rounding to E5M2: the random draws are a second input
            rb = W.random_bits16((a.rows, a.cols), seed=11, device=dev)
            ms = _time(lambda: mx.quantize(x, "e5m2", a.axis, rand=rb), a.reps,
                       _flush(a.flush, dev))
            bpe += 2.0
        else:
            ms = _time(lambda: mx.quantize(x, "e4m3", a.axis), a.reps, _flush(a.flush, dev))
        print(f"quantize {a.rows}x{a.cols} {a.axis}{' sr' if a.sr else ''}"
              f"{' fp32' if a.fp32 else ''}: {ms:.4f} ms, "
              f"{a.rows * a.cols * bpe / ms / 1e6:.1f} GB/s")
    elif a.case == "moe_quantize":
        # the routed tokens [tokens, k], per-expert groups: rowwise (forward
        # operand) or columnwise into 128-padded token segments (weight
        # gradient operand)
        x, _, offsets = W.moe_inputs(a.tokens, a.experts, a.k, 128, device=dev)
        d_off = torch.from_numpy(offsets).to(dev)
        if a.axis == "col":
            ldq = mx.mx_grouped_cols_capacity(a.tokens, a.experts)
            fn = lambda: mx.quantize_grouped(x, d_off, "e4m3", axis="col", ldq=ldq)  # noqa: E731
        else:
            fn = lambda: mx.quantize_grouped(x, d_off, "e4m3")  # noqa: E731
        ms = _time(fn, a.reps)
        print(f"moe_quantize {a.tokens}x{a.k} {a.axis} ({a.experts} experts): {ms:.4f} ms, "
              f"{a.tokens * a.k * 3.03125 / ms / 1e6:.1f} GB/s")
    elif a.case in ("moe_dgrad", "moe_wgrad"):
        # mixture-of-experts backward, FP32 out: dX_g = dY_g W_g^T or dW_g = dY_g^T X_g
        x, w, offsets = W.moe_inputs(a.tokens, a.experts, a.k, 2048, device=dev)
        e, n, k = w.shape
        dy = W.moe_grad_output(a.tokens, n, device=dev)
        d_off = torch.from_numpy(offsets).to(dev)
        if a.case == "moe_dgrad":
            qa = mx.quantize_grouped(dy, d_off, "e5m2")
            qb = mx.quantize(w.view(e * n, k), "e4m3", "col")
            y = torch.empty((a.tokens, k), dtype=torch.float32, device=dev)
            fn = lambda: mx.grouped_gemm_bcat(qa, d_off, qb, "fp32", out=y)  # noqa: E731
        else:
            ldq = mx.mx_grouped_cols_capacity(a.tokens, e)
            qa = mx.quantize_grouped(dy, d_off, "e5m2", axis="col", ldq=ldq)
            qb = mx.quantize_grouped(x, d_off, "e4m3", axis="col", ldq=ldq)
            y = torch.empty((e, n, k), dtype=torch.float32, device=dev)
            fn = lambda: mx.grouped_gemm_wgrad(qa, d_off, qb, a.tokens, "fp32", out=y)  # noqa: E731
        del x, w, dy
        ms = _time(fn, a.reps)
        print(f"{a.case} {a.tokens} tokens x {a.experts} experts ({n}x{k}): {ms:.4f} ms, "
              f"{2 * a.tokens * n * k / ms / 1e9:.1f} TFLOP/s")
    else:
        x, w, offsets = W.moe_inputs(a.tokens, a.experts, a.k, 2048, device=dev)
        e, n, k = w.shape
        d_off = torch.from_numpy(offsets).to(dev)
        qa = mx.quantize_grouped(x, d_off, "e4m3")
        qw = mx.quantize(w.view(e * n, k), "e4m3", "row")
        qb = mx.MxTensor(qw.codes.view(e, n, k), qw.scales, "e4m3")
        ms = _time(lambda: mx.grouped_gemm(qa, d_off, qb, "bf16"), a.reps)
        print(f"grouped {a.tokens} tokens x {a.experts} experts ({n}x{k}): {ms:.4f} ms, "
              f"{2 * a.tokens * n * k / ms / 1e9:.1f} TFLOP/s")
    assert mx.device_status() == 0
    return 0


if __name__ == "__main__":
    sys.exit(main())
