"""GPU parity of a blocked axis that is not a multiple of 32: the final block
holds 16 elements and is the zero-padded partial block of "Scale ownership
and the GEMM dataflow".  Quantization (codes and scales bit for bit) and the
dense, fused and grouped GEMMs (within the stated bound) against the
oracle, which completes the final block with zeros."""
import numpy as np
import pytest
import torch

from mxcheck import assert_gemm_close, ensure_built, mx_from_oracle, to_f64
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu

CONTAINER = {"e2m3", "e3m2", "e2m1"}


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def data(rows, cols, seed, dtype=torch.bfloat16):
    """N(0, 1) with per-row magnitudes spread over many binades and a few
    large entries, so that the final blocks' scales differ from their
    neighbours'."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp2(torch.randint(-8, 8, (rows, 1), generator=g).float())
    idx = torch.randperm(rows * cols, generator=g)[:max(1, rows * cols // 200)]
    x.view(-1)[idx] *= 500.0
    return x.to(dtype)


def want_codes(ref, fmt):
    return O.pack_container(ref.codes, fmt) if fmt in CONTAINER else ref.codes


def check(q, x, fmt, axis, rule="floor", rand=None):
    ref = O.quantize(to_f64(x), fmt, axis, rule, rand=rand)
    assert torch.equal(q.codes.cpu(), torch.from_numpy(want_codes(ref, fmt))), (fmt, axis)
    assert np.array_equal(q.scales.cpu().numpy(), O.swizzle_scales(ref.scales)), (fmt, axis)
    return ref


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m3", "e2m1"])
@pytest.mark.parametrize("shape", [(7, 16), (130, 48), (257, 208), (64, 1040)])
def test_rowwise_partial_final_block(mx, dtype, fmt, shape):
    x = data(*shape, seed=shape[0] + shape[1], dtype=dtype)
    for rule in ("floor", "ceil"):
        q = mx.quantize(x.cuda(), fmt, "row", rule)
        assert mx.device_status() == 0
        check(q, x, fmt, "row", rule)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", ["e4m3", "e3m2"])
@pytest.mark.parametrize("shape", [(16, 64), (48, 200), (272, 96)])
def test_colwise_partial_final_block(mx, dtype, fmt, shape):
    x = data(*shape, seed=shape[0] * 3 + shape[1], dtype=dtype)
    check(mx.quantize(x.cuda(), fmt, "col"), x, fmt, "col")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_both_orientations_with_partial_blocks_and_sr(mx, dtype):
    """Rows and columns both 16 past a multiple of 32, from one read, with
    round to nearest even and with stochastic rounding."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x = data(272, 208, seed=5, dtype=dtype)
    rand = W.random_bits16((272, 208), seed=6)
    rnp = rand.numpy().view(np.uint16).astype(np.int64)
    for fmt in ("e4m3", "e2m1"):
        row, col = mx.quantize(x.cuda(), fmt, "both")
        check(row, x, fmt, "row")
        check(col, x, fmt, "col")
        row, col = mx.quantize(x.cuda(), fmt, "both", rand=rand.cuda())
        check(row, x, fmt, "row", rand=rnp)
        check(col, x, fmt, "col", rand=rnp)
    assert mx.device_status() == 0


def test_partial_block_codes_do_not_spill_past_the_row(mx):
    """Rowwise K = 48: the final block writes only its 16 codes, so code rows
    written back to back neither overlap nor run past the buffer."""
    x = data(40, 48, seed=8)
    h = int(torch.cuda.current_stream().cuda_stream)
    s = torch.empty(mx.mx_scale_bytes(40, 48), dtype=torch.uint8, device="cuda")
    xd = x.cuda()
    # rows of 48 codes back to back, then 16 guard bytes: a final block
    # that wrote 32 codes would overwrite the next row's first 16 (caught
    # by the comparison) or, for the last row, the guard
    compact = torch.full((40 * 48 + 16,), 0xAB, dtype=torch.uint8, device="cuda")
    st = mx.mx_quantize(xd.data_ptr(), 0, 40, 48, 48, 0, 1, 0, compact.data_ptr(), s.data_ptr(),
                        None, None, h)
    assert st == 0 and mx.device_status() == 0
    assert torch.all(compact[40 * 48:].cpu() == 0xAB)
    ref = O.quantize(to_f64(x), "e4m3", "row")
    assert torch.equal(compact[:40 * 48].view(40, 48).cpu(), torch.from_numpy(ref.codes))


@pytest.mark.parametrize("k", [16, 48, 208, 7184])
@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e2m1", "e3m2")])
def test_gemm_with_partial_final_block(mx, k, fa, fb):
    """X [200, k] rowwise in fa, W [k, 264] columnwise in fb, both quantized
    on the GPU; the GEMM over the zero-padded final block matches the
    oracle's block sum."""
    m, n = 200, 264
    x = data(m, k, seed=k)
    g = torch.Generator().manual_seed(k + 1)
    w = (torch.randn(k, n, generator=g) * 0.05).to(torch.bfloat16)
    qa = mx.quantize(x.cuda(), fa, "row")
    qb = mx.quantize(w.cuda(), fb, "col")
    a = check(qa, x, fa, "row")
    b = check(qb, w, fb, "col")
    y_ref, t_ref = O.gemm(a, b)
    for out in ("fp32", "bf16"):
        y = mx.gemm(qa, qb, out)
        assert mx.device_status() == 0
        assert_gemm_close(y, y_ref, t_ref, out)


def test_gemm_on_oracle_operands_with_partial_block(mx):
    """Oracle codes with non-uniform per-block scales, K = 80: pins that the
    final block's scale is applied to its 16 products."""
    rng = np.random.default_rng(80)
    t = O.decode_table("e4m3")
    finite = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    a = O.MxBlocks(rng.choice(finite, size=(130, 80)),
                   rng.integers(118, 136, size=(130, 3)).astype(np.uint8), O.FORMATS["e4m3"])
    b = O.MxBlocks(rng.choice(finite, size=(136, 80)),
                   rng.integers(118, 136, size=(136, 3)).astype(np.uint8), O.FORMATS["e4m3"])
    y_ref, t_ref = O.gemm(a, b)
    y = mx.gemm(mx_from_oracle(a), mx_from_oracle(b), "fp32")
    assert mx.device_status() == 0
    assert_gemm_close(y, y_ref, t_ref, "fp32")


def test_fused_epilogue_with_partial_block(mx):
    m, n, k = 256, 384, 1040
    x = data(m, k, seed=3)
    g = torch.Generator().manual_seed(4)
    w = (torch.randn(k, n, generator=g) * 0.05).to(torch.bfloat16)
    bias = torch.randn(n, generator=g)
    qa, qb = mx.quantize(x.cuda(), "e4m3", "row"), mx.quantize(w.cuda(), "e4m3", "col")
    y = mx.gemm(qa, qb, "fp32", bias=bias.cuda(), act="silu")
    assert mx.device_status() == 0
    a = O.quantize(to_f64(x), "e4m3", "row")
    b = O.quantize(to_f64(w), "e4m3", "col")
    out, z, t = O.gemm_bias_act(a, b, bias.double().numpy(), "silu")
    # the bound of the dense GEMM carried through SiLU (|SiLU'| <= 1.1) plus
    # a few FP32 ulp of the add and the activation
    err = np.abs(y.cpu().double().numpy() - out)
    assert np.all(err <= 1.1e-4 * t + 2.0 ** -20 * (np.abs(z) + np.abs(out)))


def test_grouped_gemm_with_partial_block(mx):
    sizes = [0, 1, 31, 200, 0, 128, 129, 5]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    groups, total, n, k = len(sizes), int(offsets[-1]), 256, 208
    x = data(total, k, seed=11)
    g = torch.Generator().manual_seed(12)
    w = (torch.randn(groups, n, k, generator=g) * 0.02).to(torch.bfloat16)
    d_off = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(x.cuda(), d_off, "e4m3")
    qw = mx.quantize(w.cuda().view(groups * n, k), "e4m3", "row")
    qb = mx.MxTensor(qw.codes.view(groups, n, k), qw.scales, "e4m3")
    y = mx.grouped_gemm(qa, d_off, qb, "fp32")
    assert mx.device_status() == 0
    a = O.quantize(to_f64(x), "e4m3", "row")
    assert torch.equal(qa.codes.cpu(), torch.from_numpy(a.codes))
    want = O.swizzle_scales_grouped(a.scales, offsets)
    assert np.array_equal(qa.scales.cpu().numpy()[:want.size], want)
    bs = [O.quantize(to_f64(w[e]), "e4m3", "row") for e in range(groups)]
    y_ref, t_ref = O.grouped_gemm(a, offsets, bs)
    assert_gemm_close(y, y_ref, t_ref, "fp32")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_grouped_quantize_both_with_partial_row_blocks(mx, dtype):
    """Expert-grouped tokens with 208 columns (a 16-column final rowwise
    block), both orientations from one read: rowwise codes and per-group
    padded scales, and the per-expert columnwise operand, against the
    oracle."""
    sizes = [0, 1, 31, 200, 0, 128, 129, 5]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    total, cols = int(offsets[-1]), 208
    x = data(total, cols, seed=21, dtype=dtype)
    d_off = torch.from_numpy(offsets).cuda()
    ldq = mx.mx_grouped_cols_capacity(total, len(sizes))
    row, col = mx.quantize_grouped(x.cuda(), d_off, "e4m3", axis="both", ldq=ldq)
    assert mx.device_status() == 0
    ref = O.quantize(to_f64(x), "e4m3", "row")
    assert torch.equal(row.codes.cpu(), torch.from_numpy(ref.codes))
    want = O.swizzle_scales_grouped(ref.scales, offsets)
    assert np.array_equal(row.scales.cpu().numpy()[:want.size], want)
    qs = O.quantize_grouped_cols(to_f64(x), offsets, "e4m3")
    codes, scales = O.pack_grouped_cols(qs, offsets, ldq)
    used = int(O.grouped_scale_rows(offsets)[-1])
    assert torch.equal(col.codes[:, :used].cpu(), torch.from_numpy(codes[:, :used]))
    got = O.unswizzle_scales(col.scales.cpu().numpy(), cols, ldq // 32)
    assert np.array_equal(got[:, :used // 32], scales[:, :used // 32])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", ["e5m2", "e2m1", "e3m2"])
def test_rowwise_sr_with_partial_block(mx, dtype, fmt):
    """The rowwise-only stochastic-rounding pass (its own thread layout,
    and 128-column tiles for FP32) on 208 columns: a 16-column final block
    in the last tile."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x = data(130, 208, seed=17, dtype=dtype)
    rand = W.random_bits16((130, 208), seed=18)
    q = mx.quantize(x.cuda(), fmt, "row", rand=rand.cuda())
    assert mx.device_status() == 0
    check(q, x, fmt, "row", rand=rand.numpy().view(np.uint16).astype(np.int64))
