"""GPU parity of the grouped (mixture-of-experts) path: mx_quantize_grouped
plus mx_grouped_gemm against a per-group dense oracle GEMM."""
import numpy as np
import pytest
import torch

from mxcheck import assert_gemm_close, canonical_scales, ensure_built, oracle_quant, to_f64
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def run_grouped(mx, sizes, n, k, out, seed=0, fa="e4m3", fb="e4m3"):
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    groups, total = len(sizes), int(offsets[-1])
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(total, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(groups, n, k, generator=g) * 0.02).to(torch.bfloat16)
    d_off = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(x.cuda(), d_off, fa)
    qw = mx.quantize(w.cuda().view(groups * n, k), fb, "row")
    qb = mx.MxTensor(qw.codes.view(groups, n, k), qw.scales, fb)
    # guard rows after the output must stay untouched
    tdtype = torch.float32 if out == "fp32" else torch.bfloat16
    buf = torch.full((total + 8, n), float("nan"), dtype=tdtype, device="cuda")
    y = mx.grouped_gemm(qa, d_off, qb, out, out=buf[:total])
    assert mx.device_status() == 0
    assert torch.isnan(buf[total:].float()).all()
    a, _ = oracle_quant(x, fa, "row")
    assert torch.equal(qa.codes.cpu(), torch.from_numpy(a.codes))
    want = O.swizzle_scales_grouped(a.scales, offsets)
    assert np.array_equal(qa.scales.cpu().numpy()[:want.size], want)
    bs = [O.quantize(to_f64(w[e]), fb, "row") for e in range(groups)]
    y_ref, t_ref = O.grouped_gemm(a, offsets, bs)
    assert_gemm_close(y, y_ref, t_ref, out)


@pytest.mark.parametrize("sizes", [[0, 1, 31, 200, 0, 128, 129, 5], [300], [0, 0, 77],
                                   [1] * 9, [256, 0, 384]])
def test_grouped_gemm_matches_oracle(mx, sizes):
    run_grouped(mx, sizes, 256, 256, "bf16", seed=len(sizes))


def test_grouped_gemm_fp32_long_k(mx):
    run_grouped(mx, [0, 3, 130, 64, 0, 250], 384, 1056, "fp32", seed=7)


def test_grouped_gemm_e5m2_operands(mx):
    run_grouped(mx, [40, 0, 100], 128, 160, "fp32", seed=9, fa="e5m2", fb="e4m3")


def test_grouped_gemm_rejects_bad_offsets_on_device(mx):
    k, n = 64, 128
    x = torch.randn(64, k, device="cuda").to(torch.bfloat16)
    w = torch.randn(2 * n, k, device="cuda").to(torch.bfloat16)
    good = torch.tensor([0, 32, 64], dtype=torch.int32, device="cuda")
    qa = mx.quantize_grouped(x, good, "e4m3")
    qw = mx.quantize(w, "e4m3", "row")
    qb = mx.MxTensor(qw.codes.view(2, n, k), qw.scales, "e4m3")
    y = torch.zeros(64, n, device="cuda", dtype=torch.bfloat16)
    for bad in ([0, 40, 30], [1, 32, 64], [0, 32, 63]):
        mx.grouped_gemm(qa, torch.tensor(bad, dtype=torch.int32, device="cuda"), qb, out=y)
        assert mx.device_status() == 6
        assert int(y.float().abs().sum()) == 0
    mx.grouped_gemm(qa, good, qb, out=y)
    assert mx.device_status() == 0


def test_moe_full_size_sampled(mx):
    """64 experts, K=7168, N=2048, 65536 routed tokens with a Zipf(1.1)
    split including empty and sub-32-row groups; BF16 out.  Every group is
    checked on sampled rows (all rows of groups under 8 rows) and sampled
    output columns."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w, offsets = W.moe_inputs(device="cuda")
    experts, n, k = w.shape
    d_off = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(x, d_off, "e4m3")
    qw = mx.quantize(w.view(experts * n, k), "e4m3", "row")
    qb = mx.MxTensor(qw.codes.view(experts, n, k), qw.scales, "e4m3")
    y = mx.grouped_gemm(qa, d_off, qb, "bf16")
    assert mx.device_status() == 0
    sizes = np.diff(offsets)
    assert (sizes == 0).sum() >= 2 and ((sizes > 0) & (sizes < 32)).sum() >= 2
    rng = np.random.default_rng(0)
    cols = np.unique(np.concatenate([np.arange(0, 64), rng.choice(n, 64, replace=False),
                                     np.arange(n - 64, n)]))
    cols_t = torch.from_numpy(cols).cuda()
    b_scales = canonical_scales(qw.scales, experts * n, k).reshape(experts, n, k // 32)
    starts = O.grouped_scale_rows(offsets)
    for e in range(experts):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        rows = np.unique(np.concatenate([np.arange(lo, min(hi, lo + 4)),
                                         np.arange(max(lo, hi - 4), hi)]))
        rows_t = torch.from_numpy(rows).cuda()
        ra = O.quantize(to_f64(x[rows_t]), "e4m3", "row")
        assert torch.equal(qa.codes[rows_t].cpu(), torch.from_numpy(ra.codes))
        # scales of these rows inside the group's padded swizzled block
        tiles_k = -(-k // 128)
        base = starts[e] // 128 * tiles_k * 512
        part = qa.scales[base:base + O.scale_bytes(hi - lo, k // 32)].cpu().numpy()
        assert np.array_equal(O.unswizzle_scales(part, hi - lo, k // 32)[rows - lo], ra.scales)
        bq = O.quantize(to_f64(w[e][cols_t]), "e4m3", "row")
        assert torch.equal(qw.codes.view(experts, n, k)[e][cols_t].cpu(),
                           torch.from_numpy(bq.codes))
        assert np.array_equal(b_scales[e][cols], bq.scales)
        y_ref, t_ref = O.gemm(ra, bq)
        assert_gemm_close(y[rows_t][:, cols_t], y_ref, t_ref, "bf16")
