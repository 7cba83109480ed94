"""Seeded synthetic inputs for the MXFP8 matmul workloads.

This module only draws random numbers and arranges them into bf16 (or
fp32) tensors;
it holds none of the quantization or GEMM arithmetic, so both the CUDA path
and the CPU oracle can take their inputs from it.

Recipe (one reading, used everywhere):

* A value "N(0, s)" is drawn in float32 with torch's generator for the
  device it is made on, multiplied by s, then cast to bf16 (round to nearest
  even, torch's cast); an fp32 workload skips the cast.
* "p of entries replaced by +-U(lo, hi) spikes" means exactly round(p * numel)
  distinct positions (a prefix of a seeded random permutation), each set to a
  magnitude drawn from U(lo, hi) with a fair random sign, before the bf16 cast.
* Each tensor of a workload has its own seed, derived from the workload seed
  and the tensor's position, so tensors can be regenerated one at a time.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


def synth_matrix(shape, std: float, spike_frac: float = 0.0, spike_lo: float = 0.0,
                 spike_hi: float = 0.0, seed: int = 0, device="cpu",
                 dtype=torch.bfloat16) -> torch.Tensor:
    """bf16 (or `dtype`) tensor of N(0, std) with an exact count of
    +-U(lo, hi) spikes."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
    x.mul_(std)
    numel = x.numel()
    count = int(round(spike_frac * numel))
    if count:
        idx = torch.randperm(numel, generator=g, device=dev)[:count]
        mag = torch.rand(count, generator=g, device=dev, dtype=torch.float32)
        mag = mag * (spike_hi - spike_lo) + spike_lo
        sign = torch.randint(0, 2, (count,), generator=g, device=dev).to(torch.float32) * 2 - 1
        x.view(-1)[idx] = mag * sign
        del idx
    return x.to(dtype)


def random_bits16(shape, seed: int = 0, device="cpu") -> torch.Tensor:
    """Uniform 16-bit random integers (stored as int16 bit patterns), one per
    element, as the random draws of stochastic rounding."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    r = torch.randint(0, 1 << 16, tuple(shape), generator=g, device=dev, dtype=torch.int32)
    return r.to(torch.int16)


# --------------------------------------------------------------------------
# Workloads of the MXFP8 training matmul (shapes and distributions)
# --------------------------------------------------------------------------


def pr1_reference(device="cpu", seed: int = 0):
    """Small parity case: X 256x512 N(0,1) with 1% spikes +-U(200,600) and
    row 0 scaled by 1e-3 (after the spikes); W 512x256 N(0, 0.02)."""
    m, n, k = 256, 256, 512
    x = synth_matrix((m, k), 1.0, 0.01, 200.0, 600.0, seed=seed * 100 + 1, device=device)
    x = x.float()
    x[0] *= 1e-3
    x = x.to(torch.bfloat16)
    w = synth_matrix((k, n), 0.02, seed=seed * 100 + 2, device=device)
    return x, w


def quantize_sweep(shape, seed: int, device="cpu", dtype=torch.bfloat16):
    """Quantize bandwidth input: N(0,1) with 0.1% outliers +-U(100, 1e4)."""
    return synth_matrix(shape, 1.0, 0.001, 100.0, 1e4, seed=seed * 100 + 3, device=device,
                        dtype=dtype)


def dense_forward(m=16384, n=18432, k=7168, seed: int = 0, device="cpu"):
    """Forward GEMM input: X [m,k] N(0,1) with 0.5% spikes +-U(50,500);
    W [k,n] N(0,0.02)."""
    x = synth_matrix((m, k), 1.0, 0.005, 50.0, 500.0, seed=seed * 100 + 4, device=device)
    w = synth_matrix((k, n), 0.02, seed=seed * 100 + 5, device=device)
    return x, w


def dense_grad_output(m=16384, n=18432, seed: int = 0, device="cpu"):
    """Backward input dY [m,n]: N(0, 1e-3) with 0.01% spikes +-U(0.1, 1)."""
    return synth_matrix((m, n), 1e-3, 0.0001, 0.1, 1.0, seed=seed * 100 + 6, device=device)


def moe_group_sizes(total: int = 65536, experts: int = 64, seed: int = 0,
                    zipf_s: float = 1.1) -> np.ndarray:
    """Tokens per expert: multinomial over a Zipf(s) law on expert ranks
    1..E, ranks assigned to experts by a seeded permutation; then the four
    smallest groups are forced to 0, 0, 1 and 31 rows (their tokens go to the
    largest group) so that empty and sub-block groups always occur."""
    rng = np.random.default_rng(seed)
    ranks = np.arange(1, experts + 1, dtype=np.float64)
    p = ranks ** (-zipf_s)
    p /= p.sum()
    counts_by_rank = rng.multinomial(total, p)
    perm = rng.permutation(experts)
    sizes = np.empty(experts, dtype=np.int64)
    sizes[perm] = counts_by_rank
    if experts >= 5:
        order = np.argsort(sizes, kind="stable")
        forced = [0, 0, 1, 31]
        freed = 0
        for idx, v in zip(order[:4], forced):
            freed += sizes[idx] - v
            sizes[idx] = v
        sizes[np.argmax(sizes)] += freed
    assert sizes.sum() == total and (sizes >= 0).all()
    return sizes


def moe_offsets(sizes) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(sizes, dtype=np.int64))]).astype(np.int32)


def moe_inputs(total=65536, experts=64, k=7168, n=2048, seed: int = 0, device="cpu"):
    """Routed tokens X [total, k] N(0,1) (concatenated by expert) and expert
    weights stored as [experts, n, k] (each expert's W^T, K contiguous)
    N(0, 0.02)."""
    sizes = moe_group_sizes(total, experts, seed)
    x = synth_matrix((total, k), 1.0, seed=seed * 100 + 7, device=device)
    w = synth_matrix((experts, n, k), 0.02, seed=seed * 100 + 8, device=device)
    return x, w, moe_offsets(sizes)


def moe_grad_output(total=65536, n=2048, seed: int = 0, device="cpu"):
    """Output gradient of the routed tokens dY [total, n] (concatenated by
    expert): the dense backward recipe, N(0, 1e-3) with 0.01% spikes
    +-U(0.1, 1)."""
    return synth_matrix((total, n), 1e-3, 0.0001, 0.1, 1.0, seed=seed * 100 + 9, device=device)


@dataclass(frozen=True)
class GemmShape:
    m: int
    n: int
    k: int

    @property
    def flops(self) -> int:
        return 2 * self.m * self.n * self.k


FORWARD = GemmShape(16384, 18432, 7168)
DGRAD = GemmShape(16384, 7168, 18432)
WGRAD = GemmShape(7168, 18432, 16384)
