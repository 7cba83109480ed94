"""GPU parity of the MXFP6 (E2M3, E3M2) and MXFP4 (E2M1) operands: the
quantizer writes the 16-element container layout byte for byte like the
oracle, and the block-scaled GEMM on such operands (alone or mixed with
FP8) matches the oracle's block sum."""
import numpy as np
import pytest
import torch

from mxcheck import assert_gemm_close, canonical_scales, ensure_built, to_f64
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu

NARROW = ["e2m3", "e3m2", "e2m1"]


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def inputs(rows, cols, seed):
    """bf16 N(0,1) with spikes, exact zeros, negative zeros and bf16
    subnormals, so every branch of the encoders is exercised."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g)
    idx = torch.randperm(rows * cols, generator=g)
    n = rows * cols // 50
    x.view(-1)[idx[:n]] *= 1000.0
    x.view(-1)[idx[n:2 * n]] = 0.0
    x.view(-1)[idx[2 * n:3 * n]] = -0.0
    x.view(-1)[idx[3 * n:4 * n]] *= 1e-39
    x[:, :32] *= 1e-3                      # a column band of small blocks
    return x.to(torch.bfloat16)


def check_codes(q, x, fmt, axis, rule="floor"):
    ref = O.quantize(to_f64(x), fmt, axis, rule)
    want = O.pack_container(ref.codes, fmt)
    assert torch.equal(q.codes.cpu(), torch.from_numpy(want))
    rows, k = ref.codes.shape
    assert np.array_equal(canonical_scales(q.scales, rows, k), ref.scales)
    return ref


@pytest.mark.parametrize("fmt", NARROW)
@pytest.mark.parametrize("shape", [(256, 512), (288, 352), (32, 96)])
@pytest.mark.parametrize("rule", ["floor", "ceil"])
def test_narrow_quantize_matches_oracle(mx, fmt, shape, rule):
    x = inputs(*shape, seed=shape[0] + shape[1])
    row, col = mx.quantize(x.cuda(), fmt, "both", rule=rule)
    assert mx.device_status() == 0
    check_codes(row, x, fmt, "row", rule)
    check_codes(col, x, fmt, "col", rule)
    only_row = mx.quantize(x.cuda(), fmt, "row", rule=rule)
    only_col = mx.quantize(x.cuda(), fmt, "col", rule=rule)
    assert torch.equal(only_row.codes, row.codes) and torch.equal(only_col.codes, col.codes)
    assert torch.equal(only_row.scales, row.scales) and torch.equal(only_col.scales, col.scales)


@pytest.mark.parametrize("fmt", NARROW)
def test_narrow_nan_and_inf_blocks(mx, fmt):
    x = inputs(64, 128, seed=4).float()
    x[3, 40] = float("nan")
    x[10, 70] = float("inf")
    x[45, 100] = float("-inf")
    x = x.to(torch.bfloat16)
    row, col = mx.quantize(x.cuda(), fmt, "both")
    assert mx.device_status() == 0
    r = check_codes(row, x, fmt, "row")
    c = check_codes(col, x, fmt, "col")
    assert (r.scales == 0xFF).sum() == 3 and (c.scales == 0xFF).sum() == 3


@pytest.mark.parametrize("fa,fb", [("e2m1", "e2m1"), ("e2m3", "e3m2"), ("e4m3", "e2m1"),
                                   ("e3m2", "e5m2"), ("e2m1", "e4m3")])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_narrow_gemm_matches_oracle(mx, fa, fb, out):
    """X [m, k] rowwise in fa, W [k, n] columnwise in fb, on the GPU; the
    codes match the oracle and the GEMM matches the oracle's block sum."""
    m, n, k = 200, 264, 544
    x = inputs(m, k, seed=11)
    g = torch.Generator().manual_seed(12)
    w = (torch.randn(k, n, generator=g) * 0.05).to(torch.bfloat16)
    qa = mx.quantize(x.cuda(), fa, "row")
    qb = mx.quantize(w.cuda(), fb, "col")
    y = mx.gemm(qa, qb, out)
    assert mx.device_status() == 0
    a = check_codes(qa, x, fa, "row")
    b = check_codes(qb, w, fb, "col")
    y_ref, t_ref = O.gemm(a, b)
    assert_gemm_close(y, y_ref, t_ref, out)


def test_mxfp4_weights_full_size_sampled(mx):
    """Forward layer 16384 x 18432 x 7168 with E4M3 activations and MXFP4
    (E2M1) weights, BF16 out; sampled rows and columns against the oracle."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w = W.dense_forward(device="cuda")
    qa = mx.quantize(x, "e4m3", "row")
    qb = mx.quantize(w, "e2m1", "col")
    y = mx.gemm(qa, qb, "bf16")
    assert mx.device_status() == 0
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 16383], rng.choice(16384, 13, replace=False)]))
    cols = np.unique(np.concatenate([[0, 18431], rng.choice(18432, 30, replace=False)]))
    rows_t, cols_t = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    a = O.quantize(to_f64(x[rows_t]), "e4m3", "row")
    b = O.quantize(to_f64(w[:, cols_t]), "e2m1", "col")
    assert torch.equal(qb.codes[cols_t].cpu(), torch.from_numpy(O.pack_container(b.codes, "e2m1")))
    y_ref, t_ref = O.gemm(a, b)
    assert_gemm_close(y[rows_t][:, cols_t], y_ref, t_ref, "bf16")


# ---------------------------------------------------------------- packed storage

PACKED = ["e2m3_packed", "e3m2_packed", "e2m1_packed"]


def base_fmt(fmt):
    return fmt.replace("_packed", "")


def check_packed(q, x, fmt, axis, rule="floor"):
    ref = O.quantize(to_f64(x), base_fmt(fmt), axis, rule)
    want = O.pack_dense(ref.codes, base_fmt(fmt))
    assert torch.equal(q.codes.cpu(), torch.from_numpy(want))
    rows, k = ref.codes.shape
    assert np.array_equal(canonical_scales(q.scales, rows, k), ref.scales)
    return ref


@pytest.mark.parametrize("fmt", PACKED)
@pytest.mark.parametrize("shape", [(256, 512), (288, 352), (32, 96)])
@pytest.mark.parametrize("rule", ["floor", "ceil"])
def test_packed_quantize_matches_oracle(mx, fmt, shape, rule):
    """Packed 6- and 4-bit storage (K * w / 8 bytes per code row), both
    orientations, bit-exact against the oracle's dense packing; the same
    codes as the container layout with its padding removed."""
    x = inputs(*shape, seed=shape[0] * 3 + shape[1])
    row, col = mx.quantize(x.cuda(), fmt, "both", rule=rule)
    assert mx.device_status() == 0
    assert row.k == shape[1] and col.k == shape[0]
    check_packed(row, x, fmt, "row", rule)
    check_packed(col, x, fmt, "col", rule)
    only_row = mx.quantize(x.cuda(), fmt, "row", rule=rule)
    only_col = mx.quantize(x.cuda(), fmt, "col", rule=rule)
    assert torch.equal(only_row.codes, row.codes) and torch.equal(only_col.codes, col.codes)
    cont = mx.quantize(x.cuda(), base_fmt(fmt), "row", rule=rule)
    w = 4 if fmt == "e2m1_packed" else 6
    runs = cont.codes.view(shape[0], -1, 16)[:, :, :2 * w].reshape(shape[0], -1)
    assert torch.equal(runs, row.codes)
    assert torch.equal(cont.scales, row.scales)


@pytest.mark.parametrize("fa,fb", [("e2m1_packed", "e2m1_packed"), ("e4m3", "e2m1_packed"),
                                   ("e2m3_packed", "e3m2_packed"), ("e3m2_packed", "e5m2"),
                                   ("e2m1_packed", "e3m2")])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_packed_gemm_matches_oracle(mx, fa, fb, out):
    """GEMM on packed operands (read through the unpacking tensor copy):
    the oracle's block sum within the bound, and bit for bit the result of
    the same codes in the container layout."""
    m, n, k = 200, 264, 640
    x = inputs(m, k, seed=21)
    g = torch.Generator().manual_seed(22)
    w = (torch.randn(k, n, generator=g) * 0.05).to(torch.bfloat16)
    qa = mx.quantize(x.cuda(), fa, "row")
    qb = mx.quantize(w.cuda(), fb, "col")
    y = mx.gemm(qa, qb, out)
    assert mx.device_status() == 0
    a = O.quantize(to_f64(x), base_fmt(fa), "row")
    b = O.quantize(to_f64(w), base_fmt(fb), "col")
    y_ref, t_ref = O.gemm(a, b)
    assert_gemm_close(y, y_ref, t_ref, out)
    y_cont = mx.gemm(mx.quantize(x.cuda(), base_fmt(fa), "row"),
                     mx.quantize(w.cuda(), base_fmt(fb), "col"), out)
    assert torch.equal(y, y_cont)


def test_packed_mxfp4_weights_full_size_sampled(mx):
    """Forward layer 16384 x 18432 x 7168 with E4M3 activations and MXFP4
    weights in packed storage (half the container's weight bytes), BF16 out;
    sampled rows and columns against the oracle."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w = W.dense_forward(device="cuda")
    qa = mx.quantize(x, "e4m3", "row")
    qb = mx.quantize(w, "e2m1_packed", "col")
    assert qb.codes.shape == (18432, 3584)
    y = mx.gemm(qa, qb, "bf16")
    assert mx.device_status() == 0
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([[0, 16383], rng.choice(16384, 10, replace=False)]))
    cols = np.unique(np.concatenate([[0, 18431], rng.choice(18432, 20, replace=False)]))
    rows_t, cols_t = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    a = O.quantize(to_f64(x[rows_t]), "e4m3", "row")
    b = O.quantize(to_f64(w[:, cols_t]), "e2m1", "col")
    assert torch.equal(qb.codes[cols_t].cpu(), torch.from_numpy(O.pack_dense(b.codes, "e2m1")))
    y_ref, t_ref = O.gemm(a, b)
    assert_gemm_close(y[rows_t][:, cols_t], y_ref, t_ref, "bf16")


# ---------------------------------------------------------------- narrow expert weights

MOE_SIZES = [0, 1, 31, 200, 0, 128, 129, 5]


@pytest.mark.parametrize("fb", ["e2m1", "e2m1_packed", "e2m3_packed", "e3m2"])
def test_grouped_gemm_narrow_expert_weights(mx, fb):
    """Mixture-of-experts forward with E4M3 tokens and MXFP4 / MXFP6 expert
    weights, container or packed storage: every expert against the oracle's
    block sum, and packed weights equal bit for bit to the container layout
    of the same codes."""
    offsets = np.concatenate([[0], np.cumsum(MOE_SIZES)]).astype(np.int32)
    groups, total = len(MOE_SIZES), int(offsets[-1])
    n, k = 256, 384
    x = inputs(total, k, seed=31)
    g = torch.Generator().manual_seed(32)
    w = (torch.randn(groups, n, k, generator=g) * 0.05).to(torch.bfloat16)
    d_off = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(x.cuda(), d_off, "e4m3")
    qw = mx.quantize(w.cuda().view(groups * n, k), fb, "row")
    qb = mx.MxTensor(qw.codes.view(groups, n, -1), qw.scales, fb)
    y = mx.grouped_gemm(qa, d_off, qb, "fp32")
    assert mx.device_status() == 0
    a = O.quantize(to_f64(x), "e4m3", "row")
    for e in range(groups):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        be = O.quantize(to_f64(w[e]), base_fmt(fb), "row")
        y_ref, t_ref = O.gemm(O.MxBlocks(a.codes[lo:hi], a.scales[lo:hi], a.fmt), be)
        assert_gemm_close(y[lo:hi], y_ref, t_ref, "fp32")
    if fb.endswith("_packed"):
        qc = mx.quantize(w.cuda().view(groups * n, k), base_fmt(fb), "row")
        yc = mx.grouped_gemm(qa, d_off, mx.MxTensor(qc.codes.view(groups, n, k), qc.scales,
                                                    base_fmt(fb)), "fp32")
        assert torch.equal(y, yc)


@pytest.mark.parametrize("fb", ["e2m1_packed", "e2m3"])
def test_grouped_dgrad_narrow_expert_weights(mx, fb):
    """Mixture-of-experts data gradient (experts side by side along K) with
    E5M2 gradients and MXFP4 / MXFP6 expert weights quantized columnwise
    from the stacked weights, against the oracle per expert."""
    offsets = np.concatenate([[0], np.cumsum(MOE_SIZES)]).astype(np.int32)
    groups, total = len(MOE_SIZES), int(offsets[-1])
    n_model, n_expert = 264, 256
    dy = inputs(total, n_expert, seed=41)
    g = torch.Generator().manual_seed(42)
    w = (torch.randn(groups, n_expert, n_model, generator=g) * 0.02).to(torch.bfloat16)
    d_off = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(dy.cuda(), d_off, "e5m2")
    qb = mx.quantize(w.cuda().view(groups * n_expert, n_model), fb, "col")
    y = mx.grouped_gemm_bcat(qa, d_off, qb, "fp32")
    assert mx.device_status() == 0
    a = O.quantize(to_f64(dy), "e5m2", "row")
    bs = [O.quantize(to_f64(w[e]), base_fmt(fb), "col") for e in range(groups)]
    y_ref, t_ref = O.grouped_gemm(a, offsets, bs)
    assert_gemm_close(y, y_ref, t_ref, "fp32")


# ---------------------------------------------------------------- stochastic rounding

@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e3m2", "e2m1_packed", "e3m2_packed"])
@pytest.mark.parametrize("axis", ["row", "col", "both"])
def test_narrow_stochastic_rounding_matches_oracle(mx, fmt, axis):
    """MXFP4 / MXFP6 codes with stochastic rounding (container or packed
    storage): bit-exact against the oracle given the same 16-bit random
    integers, scales equal to the round-to-nearest path's."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    rows, cols = 160, 256
    x = inputs(rows, cols, seed=51)
    rand = W.random_bits16((rows, cols), seed=52)
    got = mx.quantize(x.cuda(), fmt, axis, rand=rand.cuda())
    assert mx.device_status() == 0
    rnp = rand.numpy().view(np.uint16).astype(np.int64)
    outs = got if axis == "both" else (got,)
    axes = ("row", "col") if axis == "both" else (axis,)
    pack = O.pack_dense if fmt.endswith("_packed") else O.pack_container
    for g, ax in zip(outs, axes):
        q = O.quantize(to_f64(x), base_fmt(fmt), ax, rand=rnp)
        assert torch.equal(g.codes.cpu(), torch.from_numpy(pack(q.codes, base_fmt(fmt)))), ax
        rq = O.quantize(to_f64(x), base_fmt(fmt), ax)
        assert np.array_equal(canonical_scales(g.scales, *q.codes.shape), rq.scales), ax


def test_mxfp4_stochastic_rounding_is_unbiased_on_the_gpu(mx):
    """Every element 5.5 in blocks whose amax is 6 (scale 1): over 2^16 rows
    of distinct random integers per column the GPU's E2M1 codes average to
    5.5 exactly (three quarters of the draws go up to 6)."""
    rows, cols = 1 << 16, 32
    x = torch.full((rows, cols), 5.5)
    x[:, 0] = 6.0
    r = torch.arange(rows, dtype=torch.int32).to(torch.int16).view(rows, 1).repeat(1, cols)
    q = mx.quantize(x.to(torch.bfloat16).cuda(), "e2m1", "row", rand=r.cuda().contiguous())
    assert mx.device_status() == 0
    codes = O.unpack_container(q.codes.cpu().numpy(), "e2m1")
    vals = O.decode_table("e2m1")[codes[:, 1:]]
    assert np.all(canonical_scales(q.scales, rows, cols) == 127)
    assert float(vals.mean()) == 5.5
