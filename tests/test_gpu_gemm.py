"""GPU parity of mx_gemm against the oracle.

Bound (FP32 accumulation, implementation-defined order):
|y - y_ref| <= 1e-4 * sum_k |a_hat b_hat|, plus one BF16 ulp of y_ref for
BF16 outputs.  Integer-valued cases must match bit for bit."""

import numpy as np
import pytest
import torch

from mxcheck import (assert_gemm_close, canonical_scales, ensure_built, mx_from_oracle,
                     oracle_quant, to_f64)
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def random_mx(rng, rows, k, fmt, lo=118, hi=136):
    t = O.decode_table(fmt)
    finite = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    codes = rng.choice(finite, size=(rows, k))
    scales = rng.integers(lo, hi, size=(rows, k // 32)).astype(np.uint8)
    return O.MxBlocks(codes, scales, O.FORMATS[fmt])


SHAPES = [(128, 128, 128), (256, 256, 512), (200, 136, 96), (1, 8, 32), (300, 264, 1056),
          (129, 392, 160), (64, 512, 7168)]


@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e4m3", "e5m2"),
                                   ("e5m2", "e5m2")])
def test_gemm_on_oracle_operands(mx, m, n, k, fa, fb):
    """Oracle-quantized codes with non-uniform per-block scales fed straight
    to the GPU GEMM: pins descriptors, scale layout and the block-scaled sum."""
    rng = np.random.default_rng(m * 1000 + n + k)
    a = random_mx(rng, m, k, fa)
    b = random_mx(rng, n, k, fb)
    y_ref, t_ref = O.gemm(a, b)
    for out in ("fp32", "bf16"):
        y = mx.gemm(mx_from_oracle(a), mx_from_oracle(b), out)
        assert_gemm_close(y, y_ref, t_ref, out)
    assert mx.device_status() == 0


@pytest.mark.parametrize("m,n,k", [(128, 128, 128), (256, 384, 640), (77, 136, 4096)])
def test_gemm_integer_case_is_bit_exact(mx, m, n, k):
    """Codes of small integers with power-of-two scales: every partial sum
    is an integer multiple of a power of two far below 2^24, so FP32
    accumulation is exact in any order and the GPU must match exactly."""
    rng = np.random.default_rng(k)
    av = rng.integers(-6, 7, size=(m, k)).astype(np.float64)
    bv = rng.integers(-6, 7, size=(n, k)).astype(np.float64)
    sa = rng.integers(125, 130, size=(m, k // 32)).astype(np.uint8)
    sb = rng.integers(125, 130, size=(n, k // 32)).astype(np.uint8)
    a = O.MxBlocks(O.encode_sat_rne("e4m3", av), sa, O.E4M3)
    b = O.MxBlocks(O.encode_sat_rne("e4m3", bv), sb, O.E4M3)
    y_ref, _ = O.gemm(a, b)
    y = mx.gemm(mx_from_oracle(a), mx_from_oracle(b), "fp32")
    assert np.array_equal(to_f64(y), y_ref)


def test_block_scales_stay_inside_the_sum(mx):
    """Two K-blocks with different scales (the 34-vs-25 point of the page,
    with power-of-two scale products 4 and 8): the GPU gives 2*4 + 3*8."""
    a_codes = np.zeros((128, 64), np.uint8)
    b_codes = np.zeros((128, 64), np.uint8)
    one = O.encode_sat_rne("e4m3", np.array([1.0]))[0]
    a_codes[:, 0:2] = one
    a_codes[:, 32:35] = one
    b_codes[:, :] = one
    sa = np.tile(np.array([[129, 130]], np.uint8), (128, 1))
    sb = np.full((128, 2), 127, np.uint8)
    a = O.MxBlocks(a_codes, sa, O.E4M3)
    b = O.MxBlocks(b_codes, sb, O.E4M3)
    y = to_f64(mx.gemm(mx_from_oracle(a), mx_from_oracle(b), "fp32"))
    assert np.all(y == 32.0)


def test_output_leading_dimension(mx):
    rng = np.random.default_rng(5)
    a = random_mx(rng, 160, 256, "e4m3")
    b = random_mx(rng, 136, 256, "e4m3")
    y_ref, t_ref = O.gemm(a, b)
    big = torch.full((160, 200), float("nan"), device="cuda")
    mx.gemm(mx_from_oracle(a), mx_from_oracle(b), "fp32", out=big[:, 16:152])
    assert_gemm_close(big[:, 16:152], y_ref, t_ref, "fp32")
    assert torch.isnan(big[:, :16]).all() and torch.isnan(big[:, 152:]).all()


def test_pr1_reference_end_to_end(mx):
    """The small reference configuration: X 256x512 with spikes and a 1e-3
    row, W 512x256; GPU quantize then GPU GEMM, FP32 out."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w = W.pr1_reference()
    qa = mx.quantize(x.cuda(), "e4m3", "row")
    qb = mx.quantize(w.cuda(), "e4m3", "col")
    a, _ = oracle_quant(x, "e4m3", "row")
    b, _ = oracle_quant(w, "e4m3", "col")
    assert torch.equal(qa.codes.cpu(), torch.from_numpy(a.codes))
    assert torch.equal(qb.codes.cpu(), torch.from_numpy(b.codes))
    y_ref, t_ref = O.gemm(a, b)
    y = mx.gemm(qa, qb, "fp32")
    assert_gemm_close(y, y_ref, t_ref, "fp32")


def sampled_check(mx, y, qa, qb, a_rows, b_rows, out):
    """Oracle GEMM on sampled rows of A and B (taken from the GPU-written,
    already verified codes and scales) against the GPU output block."""
    m, k = qa.codes.shape
    n = qb.codes.shape[0]
    sa = canonical_scales(qa.scales, m, k)
    sb = canonical_scales(qb.scales, n, k)
    ar, br = a_rows.cuda(), b_rows.cuda()
    a = O.MxBlocks(qa.codes[ar].cpu().numpy(), sa[a_rows.numpy()], O.FORMATS[qa.fmt])
    b = O.MxBlocks(qb.codes[br].cpu().numpy(), sb[b_rows.numpy()], O.FORMATS[qb.fmt])
    y_ref, t_ref = O.gemm(a, b)
    return assert_gemm_close(y[ar][:, br], y_ref, t_ref, out)


def stripes(total, width=128):
    mid = (total // 2) // width * width
    idx = np.concatenate([np.arange(0, width), np.arange(mid, mid + width),
                          np.arange(total - width, total)])
    return torch.from_numpy(np.unique(idx))


def test_forward_full_size_sampled(mx):
    """Dense forward M=16384, N=18432, K=7168, E4M3 x E4M3, BF16 out."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w = W.dense_forward(device="cuda")
    qa = mx.quantize(x, "e4m3", "row")
    qb = mx.quantize(w, "e4m3", "col")
    y = mx.gemm(qa, qb, "bf16")
    rows = stripes(x.shape[0])
    cols = stripes(w.shape[1])
    ra = O.quantize(to_f64(x[rows.cuda()]), "e4m3", "row")
    assert torch.equal(qa.codes[rows.cuda()].cpu(), torch.from_numpy(ra.codes))
    rb = O.quantize(to_f64(w[:, cols.cuda()]), "e4m3", "col")
    assert torch.equal(qb.codes[cols.cuda()].cpu(), torch.from_numpy(rb.codes))
    assert np.array_equal(canonical_scales(qb.scales, w.shape[1], w.shape[0])[cols], rb.scales)
    sampled_check(mx, y, qa, qb, rows, cols, "bf16")
    assert mx.device_status() == 0


def test_fused_forward_full_size_sampled(mx):
    """The fused epilogue in the bench's launch configuration: dense forward
    M=16384, N=18432, K=7168 with an FP32 bias and SiLU, BF16 out, checked on
    sampled rows and columns (GPU-written codes and scales, verified by
    test_forward_full_size_sampled) against the oracle's epilogue."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w = W.dense_forward(device="cuda")
    qa = mx.quantize(x, "e4m3", "row")
    qb = mx.quantize(w, "e4m3", "col")
    del x, w
    n = qb.codes.shape[0]
    bias = torch.randn(n, generator=torch.Generator().manual_seed(21)) * 0.5
    y = mx.gemm(qa, qb, "bf16", bias=bias.cuda(), act="silu")
    assert mx.device_status() == 0
    m, k = qa.codes.shape
    rows, cols = stripes(m), stripes(n)
    sa = canonical_scales(qa.scales, m, k)
    sb = canonical_scales(qb.scales, n, k)
    a = O.MxBlocks(qa.codes[rows.cuda()].cpu().numpy(), sa[rows.numpy()], O.FORMATS[qa.fmt])
    b = O.MxBlocks(qb.codes[cols.cuda()].cpu().numpy(), sb[cols.numpy()], O.FORMATS[qb.fmt])
    out_ref, z_ref, t_ref = O.gemm_bias_act(a, b, bias.double().numpy()[cols.numpy()], "silu")
    r = fused_error_ratio(y[rows.cuda()][:, cols.cuda()], out_ref, z_ref, t_ref, "bf16")
    assert r <= 1.0, f"fused epilogue error {r:.3g} x bound"


def test_dgrad_and_wgrad_full_size_sampled(mx):
    """Backward GEMMs of the same layer: dgrad dX = dY W^T with dY E5M2
    (blocks along N) and W E4M3 (blocks along N); wgrad dW = X^T dY over
    K = 16384 tokens, E4M3 x E5M2; both FP32 out."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w = W.dense_forward(device="cuda")
    dy = W.dense_grad_output(device="cuda")
    # dgrad: A = dY [16384, 18432] rowwise E5M2, B = W [7168, 18432] rowwise E4M3
    qa = mx.quantize(dy, "e5m2", "row")
    qb = mx.quantize(w, "e4m3", "row")
    dx = mx.gemm(qa, qb, "fp32")
    rows = stripes(dy.shape[0])
    cols = stripes(w.shape[0])
    ra = O.quantize(to_f64(dy[rows.cuda()]), "e5m2", "row")
    assert torch.equal(qa.codes[rows.cuda()].cpu(), torch.from_numpy(ra.codes))
    sampled_check(mx, dx, qa, qb, rows, cols, "fp32")
    del dx, qa, qb
    # wgrad: A = X^T [7168, 16384] (X colwise), B = dY^T [18432, 16384] (dY colwise)
    qa = mx.quantize(x, "e4m3", "col")
    qb = mx.quantize(dy, "e5m2", "col")
    dw = mx.gemm(qa, qb, "fp32")
    rows = stripes(x.shape[1])
    cols = stripes(dy.shape[1])
    rb = O.quantize(to_f64(dy[:, cols.cuda()]), "e5m2", "col")
    assert torch.equal(qb.codes[cols.cuda()].cpu(), torch.from_numpy(rb.codes))
    sampled_check(mx, dw, qa, qb, rows, cols, "fp32")
    assert mx.device_status() == 0


def fused_error_ratio(y_gpu, out_ref, z_ref, t_ref, out_dtype):
    """Fused-epilogue bound: the GEMM bound carried through the activation
    (|silu'| <= 1.1), FP32 rounding of the add and the activation (2^-20
    relative), and one BF16 ulp for BF16 outputs."""
    from mxcheck import bf16_ulp
    y = to_f64(y_gpu)
    allowed = 1.1e-4 * t_ref + 2.0 ** -20 * (np.abs(z_ref) + np.abs(out_ref))
    if out_dtype == "bf16":
        allowed = allowed + bf16_ulp(out_ref)
    assert np.isfinite(y).all()
    return float((np.abs(y - out_ref) / np.maximum(allowed, 1e-300)).max())


@pytest.mark.parametrize("m,n,k", [(128, 256, 256), (300, 264, 1056), (77, 520, 160)])
@pytest.mark.parametrize("act", ["none", "silu"])
@pytest.mark.parametrize("with_bias", [True, False])
def test_fused_bias_act_epilogue(mx, m, n, k, act, with_bias):
    """The kernel contract's epilogue: act(acc + bias[col]) in FP32, one
    rounding to BF16 / FP32."""
    if not with_bias and act == "none":
        pytest.skip("plain GEMM")
    rng = np.random.default_rng(m + n + k)
    a = random_mx(rng, m, k, "e4m3", 118, 126)
    b = random_mx(rng, n, k, "e4m3", 118, 126)
    bias = rng.standard_normal(n).astype(np.float32) * 4 if with_bias else None
    out_ref, z_ref, t_ref = O.gemm_bias_act(a, b, None if bias is None else bias.astype(np.float64), act)
    bt = torch.from_numpy(bias).cuda() if with_bias else None
    for out in ("bf16", "fp32"):
        y = mx.gemm(mx_from_oracle(a), mx_from_oracle(b), out, bias=bt, act=act)
        r = fused_error_ratio(y, out_ref, z_ref, t_ref, out)
        assert r <= 1.0, f"fused epilogue error {r:.3g} x bound ({out})"
    assert mx.device_status() == 0


def test_fused_epilogue_rejects_grouped_and_bad_args(mx):
    assert mx.mx_gemm_bias_act(128, 128, 64, 16, 16, 0, 16, 16, 0, None, 7, 16, 0, 128, 0) == 1
    assert mx.mx_gemm_bias_act(128, 128, 64, 16, 16, 0, 16, 16, 0, 20, 1, 16, 0, 128, 0) == 2


def test_wait_timeout_selftest(mx):
    """A wait on an mbarrier that nothing completes gives up by itself and
    reports MX_ERR_TIMEOUT; the context stays usable."""
    assert mx.device_status() == 0
    assert mx.mx_selftest_wait_timeout(2_000_000) == 0     # 2 ms
    assert mx.device_status() == 5
    assert mx.device_status() == 0
    x = torch.randn(128, 128, device="cuda").to(torch.bfloat16)
    q = mx.quantize(x, "e4m3", "row")
    assert q.codes.shape == (128, 128)
    assert mx.device_status() == 0
