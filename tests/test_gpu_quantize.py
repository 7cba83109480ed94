"""GPU parity of mx_quantize / mx_quantize_grouped against the oracle.

Codes and scales must match bit for bit, including the zero padding of the
swizzled scale buffer."""
import numpy as np
import pytest
import torch

from mxcheck import (INCIDENT_LOG, canonical_scales, ensure_built, incident_counts,
                     oracle_quant, to_f64)
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def special_matrix(rows, cols, seed):
    """bf16 matrix mixing normal data with every block edge case: zeros,
    signed zeros, bf16 subnormals, equal values, binade edges, amax
    significands just above 1.75, huge and tiny magnitudes."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 4)
    flat = x.view(-1)
    nb = flat.numel() // 32
    kinds = torch.randint(0, 10, (nb,), generator=g)
    for b in range(nb):
        blk = flat[b * 32:(b + 1) * 32]
        k = int(kinds[b])
        if k == 0:
            blk.zero_()
        elif k == 1:
            blk.zero_()
            blk[::3] = -0.0
        elif k == 2:
            blk.copy_(torch.randn(32, generator=g) * 2.0 ** -130)   # bf16 subnormals
        elif k == 3:
            blk.fill_(float(torch.randn(1, generator=g)))
        elif k == 4:
            blk.mul_(0.01)
            blk[5] = 2.0 ** int(torch.randint(-20, 20, (1,), generator=g))  # amax at a binade edge
        elif k == 5:
            blk[7] = 1.8125 * 2.0 ** int(torch.randint(-20, 20, (1,), generator=g))  # sig > 1.75
        elif k == 6:
            blk.mul_(1e30)
        elif k == 7:
            blk.mul_(1e-30)
    return x.to(torch.bfloat16)


def check_row(mx, x, fmt, rule):
    rows, cols = x.shape
    got = mx.quantize(x.cuda(), fmt, "row", rule)
    q, sw = oracle_quant(x, fmt, "row", rule)
    assert torch.equal(got.codes.cpu(), torch.from_numpy(q.codes))
    assert np.array_equal(got.scales.cpu().numpy(), sw)


def check_col(mx, x, fmt, rule):
    got = mx.quantize(x.cuda(), fmt, "col", rule)
    q, sw = oracle_quant(x, fmt, "col", rule)
    assert torch.equal(got.codes.cpu(), torch.from_numpy(q.codes))
    assert np.array_equal(got.scales.cpu().numpy(), sw)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("rule", ["floor", "ceil"])
@pytest.mark.parametrize("shape", [(1, 32), (7, 96), (128, 128), (300, 416), (257, 1056)])
def test_rowwise_matches_oracle(mx, fmt, rule, shape):
    x = special_matrix(*shape, seed=shape[0] * 7 + shape[1])
    check_row(mx, x, fmt, rule)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("rule", ["floor", "ceil"])
@pytest.mark.parametrize("shape", [(32, 8), (96, 200), (128, 128), (416, 264), (1056, 136)])
def test_colwise_matches_oracle(mx, fmt, rule, shape):
    # edge-case blocks laid out along columns (the blocked axis here)
    x = special_matrix(shape[1], shape[0], seed=shape[0] * 5 + shape[1]).T.contiguous()
    check_col(mx, x, fmt, rule)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_both_from_one_read_equals_separate(mx, fmt):
    x = special_matrix(320, 480, seed=3)
    xr = x.cuda()
    r, c = mx.quantize(xr, fmt, "both")
    q, sw = oracle_quant(x, fmt, "row")
    assert torch.equal(r.codes.cpu(), torch.from_numpy(q.codes))
    assert np.array_equal(r.scales.cpu().numpy(), sw)
    q, sw = oracle_quant(x, fmt, "col")
    assert torch.equal(c.codes.cpu(), torch.from_numpy(q.codes))
    assert np.array_equal(c.scales.cpu().numpy(), sw)


def test_nan_and_inf_blocks(mx):
    x = torch.randn(64, 128)
    x[0, 3] = float("nan")
    x[5, 70] = float("inf")
    x[40, 100] = float("-inf")
    x = x.to(torch.bfloat16)
    for axis in ("row", "col"):
        got = mx.quantize(x.cuda(), "e4m3", axis)
        q, sw = oracle_quant(x, "e4m3", axis)
        assert torch.equal(got.codes.cpu(), torch.from_numpy(q.codes))
        assert np.array_equal(got.scales.cpu().numpy(), sw)
        assert (got.scales.cpu().numpy() == 0xFF).sum() == 3


def test_strided_input(mx):
    base = special_matrix(96, 320, seed=11)
    x = base[:, 64:256]          # ldx = 320 > cols = 192
    got = mx.quantize(base.cuda()[:, 64:256], "e4m3", "both")
    qr, swr = oracle_quant(x.contiguous(), "e4m3", "row")
    qc, swc = oracle_quant(x.contiguous(), "e4m3", "col")
    assert torch.equal(got[0].codes.cpu(), torch.from_numpy(qr.codes))
    assert np.array_equal(got[0].scales.cpu().numpy(), swr)
    assert torch.equal(got[1].codes.cpu(), torch.from_numpy(qc.codes))
    assert np.array_equal(got[1].scales.cpu().numpy(), swc)


def test_two_row_fixture_on_gpu_reproduces_page_scales(mx):
    """The page's two-row experiment (rows padded to 32 for the column
    kernel is not needed: rowwise only), ceil rule: scales 2^-8 and 2."""
    small = [0.001, 0.03, 0.117, 0.5, 1.0, -0.25, 0.0625, -0.015625] * 4
    large = [4.0, 16.0, 64.0, 500.0, -2.0, -8.0, -32.0, -250.0] * 4
    x = torch.tensor([small, large], dtype=torch.float32).to(torch.bfloat16)
    got = mx.quantize(x.cuda(), "e4m3", "row", "ceil")
    sc = canonical_scales(got.scales, 2, 32)
    assert [O.decode_e8m0(int(s)) for s in sc[:, 0]] == [2.0 ** -8, 2.0]
    check_row(mx, x, "e4m3", "ceil")
    check_row(mx, x, "e4m3", "floor")


@pytest.mark.parametrize("variant", ["zero_small_row", "spike_in_small_row"])
@pytest.mark.parametrize("rule", ["ceil", "floor"])
def test_troubleshooting_fixtures_on_gpu(mx, variant, rule):
    """The page's troubleshooting changes to the two-row fixture ("Troubleshooting
    numerical failures"): the small row all zeros, or 500 in the small row's
    block (x[0, 3] = 500), each projected by the original W and by a column
    selecting only the spike (padded with zero columns to n = 16).  Codes
    and scales bit-exact against the oracle; the projections are exact sums
    of a few dyadic products, so the FP32 outputs must match exactly."""
    small = [0.001, 0.03, 0.117, 0.5, 1.0, -0.25, 0.0625, -0.015625] * 4
    large = [4.0, 16.0, 64.0, 500.0, -2.0, -8.0, -32.0, -250.0] * 4
    x = torch.tensor([small, large], dtype=torch.float32)
    if variant == "zero_small_row":
        x[0] = 0.0
    else:
        x[0, 3] = 500.0
    x = x.to(torch.bfloat16)
    check_row(mx, x, "e4m3", rule)
    w = torch.zeros(32, 16)
    w[:, 1] = torch.tensor([0.5, -0.25, 0.125, -0.0625, 0.03125, -0.5, 0.25, -0.125] * 4)
    w[3, 0] = 1.0                                   # the selector
    w = w.to(torch.bfloat16)
    check_col(mx, w, "e4m3", rule)
    qx = mx.quantize(x.cuda(), "e4m3", "row", rule)
    qw = mx.quantize(w.cuda(), "e4m3", "col", rule)
    y = mx.gemm(qx, qw, "fp32").cpu().double().numpy()
    ox, _ = oracle_quant(x, "e4m3", "row", rule)
    ow, _ = oracle_quant(w, "e4m3", "col", rule)
    y_ref, _ = O.gemm(ox, ow)
    assert np.array_equal(y, y_ref)
    spike = 512.0 if rule == "ceil" else 448.0
    small_sel = 0.0 if variant == "zero_small_row" else spike
    assert y[:, 0].tolist() == [small_sel, spike]
    assert (y[:, 2:] == 0).all()
    assert mx.device_status() == 0


def test_pr1_reference_inputs(mx):
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w = W.pr1_reference()
    check_row(mx, x, "e4m3", "floor")
    check_col(mx, w, "e4m3", "floor")


def test_quantize_sweep_4096_full(mx):
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x = W.quantize_sweep((4096, 4096), seed=0, device="cuda")
    r, c = mx.quantize(x, "e4m3", "both")
    xc = x.cpu()
    q, sw = oracle_quant(xc, "e4m3", "row")
    assert torch.equal(r.codes.cpu(), torch.from_numpy(q.codes))
    assert np.array_equal(r.scales.cpu().numpy(), sw)
    q, sw = oracle_quant(xc, "e4m3", "col")
    assert torch.equal(c.codes.cpu(), torch.from_numpy(q.codes))
    assert np.array_equal(c.scales.cpu().numpy(), sw)


def test_quantize_sweep_16384x8192_sampled(mx):
    """Full-size launch; the oracle checks sampled 128-row / 128-column
    stripes (first, interior, last) of both orientations."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    rows, cols = 16384, 8192
    x = W.quantize_sweep((rows, cols), seed=1, device="cuda")
    r, c = mx.quantize(x, "e4m3", "both")
    rs = canonical_scales(r.scales, rows, cols)
    cs = canonical_scales(c.scales, cols, rows)
    for r0 in (0, 128 * 61, rows - 128):
        xs = x[r0:r0 + 128].cpu()
        q = O.quantize(to_f64(xs), "e4m3", "row")
        assert torch.equal(r.codes[r0:r0 + 128].cpu(), torch.from_numpy(q.codes))
        assert np.array_equal(rs[r0:r0 + 128], q.scales)
    for c0 in (0, 128 * 29, cols - 128):
        xs = x[:, c0:c0 + 128].cpu()
        q = O.quantize(to_f64(xs), "e4m3", "col")
        assert torch.equal(c.codes[c0:c0 + 128].cpu(), torch.from_numpy(q.codes))
        assert np.array_equal(cs[c0:c0 + 128], q.scales)


def test_grouped_rowwise_matches_oracle(mx):
    sizes = [0, 1, 31, 200, 0, 128, 129, 5]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    total, cols = int(offsets[-1]), 288
    x = special_matrix(total, cols, seed=21)
    got = mx.quantize_grouped(x.cuda(), torch.from_numpy(offsets).cuda(), "e4m3")
    q, _ = oracle_quant(x, "e4m3", "row")
    assert torch.equal(got.codes.cpu(), torch.from_numpy(q.codes))
    want = O.swizzle_scales_grouped(q.scales, offsets)
    assert np.array_equal(got.scales.cpu().numpy()[:want.size], want)


def test_grouped_quantize_rejects_bad_offsets_on_device(mx):
    x = torch.randn(64, 64).to(torch.bfloat16).cuda()
    bad = torch.tensor([0, 40, 30, 64], dtype=torch.int32).cuda()   # not monotone
    mx.device_status()
    got = mx.quantize_grouped(x, bad, "e4m3")
    assert mx.device_status() == 6
    assert int(got.scales.abs().sum()) == 0
    assert mx.device_status() == 0


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("axis", ["row", "col", "both"])
@pytest.mark.parametrize("shape", [(32, 64), (160, 224), (416, 264)])
def test_stochastic_rounding_matches_oracle(mx, fmt, axis, shape):
    """Bit-exact codes given the same 16-bit random integers; scales equal
    the round-to-nearest path's."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    rows, cols = shape
    if axis != "col" and cols % 32:
        pytest.skip("rowwise needs cols % 32 == 0")
    x = special_matrix(rows, cols, seed=rows + cols) if axis != "col" else \
        special_matrix(cols, rows, seed=rows + cols).T.contiguous()
    rand = W.random_bits16((rows, cols), seed=rows * 3 + cols)
    got = mx.quantize(x.cuda(), fmt, axis, rand=rand.cuda())
    rnp = rand.numpy().view(np.uint16).astype(np.int64)
    outs = got if axis == "both" else (got,)
    axes = ("row", "col") if axis == "both" else (axis,)
    for g, ax in zip(outs, axes):
        q = O.quantize(to_f64(x), fmt, ax, rand=rnp)
        assert torch.equal(g.codes.cpu(), torch.from_numpy(q.codes)), ax
        assert np.array_equal(g.scales.cpu().numpy(), O.swizzle_scales(q.scales)), ax


def test_stochastic_rounding_full_size_sampled(mx):
    """16384x8192 E5M2 both orientations with random draws; sampled stripes
    against the oracle, and the mean of the dequantized values tracks the
    input (unbiased rounding)."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    rows, cols = 16384, 8192
    x = W.quantize_sweep((rows, cols), seed=1, device="cuda")
    rand = W.random_bits16((rows, cols), seed=5, device="cuda")
    r, c = mx.quantize(x, "e5m2", "both", rand=rand)
    rs = canonical_scales(r.scales, rows, cols)
    for r0 in (0, rows - 128):
        xs = x[r0:r0 + 128].cpu()
        rn = rand[r0:r0 + 128].cpu().numpy().view(np.uint16).astype(np.int64)
        q = O.quantize(to_f64(xs), "e5m2", "row", rand=rn)
        assert torch.equal(r.codes[r0:r0 + 128].cpu(), torch.from_numpy(q.codes))
        assert np.array_equal(rs[r0:r0 + 128], q.scales)
    for c0 in (0, cols - 128):
        xs = x[:, c0:c0 + 128].cpu()
        rn = rand[:, c0:c0 + 128].cpu().numpy().view(np.uint16).astype(np.int64)
        q = O.quantize(to_f64(xs), "e5m2", "col", rand=rn)
        assert torch.equal(c.codes[c0:c0 + 128].cpu(), torch.from_numpy(q.codes))


@pytest.mark.parametrize("fmt,rule", [("e4m3", "floor"), ("e4m3", "ceil"), ("e5m2", "floor")])
def test_incident_trace_counts_of_gpu_output(mx, fmt, rule):
    """The incident trace's clip and zero counts read off the GPU's codes and
    scales equal the oracle's, on the forward layer's activations (2048 of
    its rows, spikes included) and the quantize sweep's 4096x4096 tensor
    (with +-U(100, 1e4) outliers), rowwise and columnwise."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x_fwd, _ = W.dense_forward(device="cuda")
    cases = [("forward X[:2048]", x_fwd[:2048].contiguous()),
             ("sweep 4096x4096", W.quantize_sweep((4096, 4096), seed=0, device="cuda"))]
    del x_fwd
    for name, x in cases:
        xc = x.cpu()
        for axis in ("row", "col"):
            q = mx.quantize(x, fmt, axis, rule=rule)
            assert mx.device_status() == 0
            got = incident_counts(xc, q.codes, q.scales, fmt, axis)
            t = O.incident_trace(to_f64(xc), fmt, axis, rule)
            assert got == (t.clip_count, t.zero_count, t.nan_blocks)
            INCIDENT_LOG.append((f"{name}", f"{name} {axis} {fmt} {rule}", xc.numel(), *got))
