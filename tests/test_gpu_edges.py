"""Degenerate and extreme sizes on the GPU: empty inputs, the smallest legal
shapes, groups that are all empty, and the largest group count, for the
quantizers and the three GEMM modes (both GEMM kernels)."""
import numpy as np
import pytest
import torch

from mxcheck import assert_gemm_close, canonical_scales, ensure_built, to_f64
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def h():
    return int(torch.cuda.current_stream().cuda_stream)


def test_empty_quantize_writes_nothing(mx):
    sentinel = torch.full((256,), 0xAB, dtype=torch.uint8, device="cuda")
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    # rows = 0 and cols = 0 are valid and launch nothing
    assert mx.mx_quantize(x.data_ptr(), 0, 0, 32, 32, 0, 3, 0, sentinel.data_ptr(),
                          sentinel.data_ptr(), sentinel.data_ptr(), sentinel.data_ptr(), h()) == 0
    assert mx.mx_quantize(x.data_ptr(), 0, 32, 0, 0, 0, 1, 0, sentinel.data_ptr(),
                          sentinel.data_ptr(), None, None, h()) == 0
    assert mx.device_status() == 0
    assert (sentinel == 0xAB).all()


@pytest.mark.parametrize("shape,axis", [((1, 32), "row"), ((32, 8), "col"), ((32, 32), "both")])
def test_smallest_quantize_shapes(mx, shape, axis):
    g = torch.Generator().manual_seed(1)
    x = (torch.randn(*shape, generator=g) * 10).to(torch.bfloat16)
    out = mx.quantize(x.cuda(), "e4m3", axis)
    assert mx.device_status() == 0
    pairs = [(out[0], "row"), (out[1], "col")] if axis == "both" else [(out, axis)]
    for q, ax in pairs:
        ref = O.quantize(to_f64(x), "e4m3", ax)
        assert torch.equal(q.codes.cpu(), torch.from_numpy(ref.codes))
        rows, k = ref.codes.shape
        assert np.array_equal(canonical_scales(q.scales, rows, k), ref.scales)


@pytest.mark.parametrize("m,n,k", [(1, 8, 32), (2, 16, 32), (1, 264, 32), (300, 8, 64)])
def test_smallest_gemm_shapes(mx, m, n, k):
    g = torch.Generator().manual_seed(m + n + k)
    x = torch.randn(m, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(k, n, generator=g) * 0.1).to(torch.bfloat16)
    qa = mx.quantize(x.cuda(), "e4m3", "row")
    qb = mx.quantize(w.cuda(), "e4m3", "col")
    for out in ("fp32", "bf16"):
        y = mx.gemm(qa, qb, out)
        assert mx.device_status() == 0
        a = O.quantize(to_f64(x), "e4m3", "row")
        b = O.quantize(to_f64(w), "e4m3", "col")
        y_ref, t_ref = O.gemm(a, b)
        assert_gemm_close(y, y_ref, t_ref, out)


def test_gemm_with_no_rows_launches_nothing(mx):
    y = torch.full((8, 8), 3.0, device="cuda")
    codes = torch.zeros(8, 32, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(512, dtype=torch.uint8, device="cuda")
    assert mx.mx_gemm(0, 8, 32, codes.data_ptr(), scales.data_ptr(), 0, codes.data_ptr(),
                      scales.data_ptr(), 0, y.data_ptr(), 1, 8, h()) == 0
    assert mx.device_status() == 0
    assert (y == 3.0).all()


def test_grouped_gemms_with_every_group_empty(mx):
    """No tokens at all: the row-grouped GEMMs write nothing, the weight
    gradient writes zeros for every expert."""
    groups, n, k = 5, 128, 128
    d_off = torch.zeros(groups + 1, dtype=torch.int32, device="cuda")
    a = torch.zeros(1, k, dtype=torch.uint8, device="cuda")
    sa = torch.zeros(mx.mx_grouped_scale_bytes(0, groups, k), dtype=torch.uint8, device="cuda")
    b = torch.zeros(groups * n, k, dtype=torch.uint8, device="cuda")
    sb = torch.zeros(groups * mx.mx_scale_bytes(n, k), dtype=torch.uint8, device="cuda")
    y = torch.full((4, n), 7.0, device="cuda")
    assert mx.mx_grouped_gemm(groups, d_off.data_ptr(), 0, n, k, a.data_ptr(), sa.data_ptr(), 0,
                              b.data_ptr(), sb.data_ptr(), 0, y.data_ptr(), 1, h()) == 0
    assert mx.device_status() == 0
    assert (y == 7.0).all()
    # weight gradient over zero tokens: [groups, m, n] of zeros
    ldq = 128
    qa = torch.zeros(256, ldq, dtype=torch.uint8, device="cuda")
    sqa = torch.zeros(mx.mx_scale_bytes(256, ldq), dtype=torch.uint8, device="cuda")
    qb = torch.zeros(n, ldq, dtype=torch.uint8, device="cuda")
    sqb = torch.zeros(mx.mx_scale_bytes(n, ldq), dtype=torch.uint8, device="cuda")
    dw = torch.full((groups, 256, n), 5.0, device="cuda")
    assert mx.mx_grouped_gemm_wgrad(groups, d_off.data_ptr(), 0, 256, n, ldq, qa.data_ptr(),
                                    sqa.data_ptr(), 1, qb.data_ptr(), sqb.data_ptr(), 0,
                                    dw.data_ptr(), 1, h()) == 0
    assert mx.device_status() == 0
    assert int((dw != 0).sum()) == 0


def test_largest_group_count(mx):
    """1000 groups (the library's maximum), most of them empty, a few with
    ragged sizes: the device group table covers them all."""
    groups, n, k = 1000, 128, 64
    sizes = np.zeros(groups, dtype=np.int64)
    rng = np.random.default_rng(8)
    sizes[rng.choice(groups, 12, replace=False)] = rng.integers(1, 200, 12)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    total = int(offsets[-1])
    g = torch.Generator().manual_seed(9)
    x = torch.randn(total, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(groups, n, k, generator=g) * 0.05).to(torch.bfloat16)
    d_off = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(x.cuda(), d_off, "e4m3")
    qw = mx.quantize(w.cuda().view(groups * n, k), "e4m3", "row")
    qb = mx.MxTensor(qw.codes.view(groups, n, k), qw.scales, "e4m3")
    y = mx.grouped_gemm(qa, d_off, qb, "fp32")
    assert mx.device_status() == 0
    a = O.quantize(to_f64(x), "e4m3", "row")
    used = [e for e in range(groups) if sizes[e]]
    for e in used:
        lo, hi = offsets[e], offsets[e + 1]
        be = O.quantize(to_f64(w[e]), "e4m3", "row")
        y_ref, t_ref = O.gemm(O.MxBlocks(a.codes[lo:hi], a.scales[lo:hi], a.fmt), be)
        assert_gemm_close(y[lo:hi], y_ref, t_ref, "fp32")


def test_buffers_beyond_2_gib_of_elements(mx):
    """Operands and outputs with more than 2^31 elements (64-bit offsets in
    every kernel): a rowwise quantize of 40960 x 57344 bf16 (2.35 G
    elements) checked on its last rows and first rows, and a GEMM whose
    65536 x 36864 output (2.4 G elements) is checked on its last rows and
    columns."""
    rows, cols = 40960, 57344
    g = torch.Generator(device="cuda").manual_seed(12)
    x = (torch.randn(rows, cols, generator=g, device="cuda") * 3).to(torch.bfloat16)
    q = mx.quantize(x, "e4m3", "row")
    assert mx.device_status() == 0
    for lo in (0, rows - 128):
        ref = O.quantize(to_f64(x[lo:lo + 128, :4096]), "e4m3", "row")
        assert torch.equal(q.codes[lo:lo + 128, :4096].cpu(), torch.from_numpy(ref.codes))
        tail = O.quantize(to_f64(x[lo:lo + 128, cols - 4096:]), "e4m3", "row")
        assert torch.equal(q.codes[lo:lo + 128, cols - 4096:].cpu(), torch.from_numpy(tail.codes))
    kb = cols // 32
    r, c = np.meshgrid(np.arange(rows - 128, rows), np.arange(kb - 128, kb), indexing="ij")
    got = q.scales.cpu().numpy()[O.swizzle_offset(r, c, kb)]
    assert np.array_equal(got, tail.scales)
    del x, q
    torch.cuda.empty_cache()
    m, n, k = 65536, 36864, 64
    a = (torch.randn(m, k, generator=g, device="cuda")).to(torch.bfloat16)
    b = (torch.randn(k, n, generator=g, device="cuda") * 0.1).to(torch.bfloat16)
    qa = mx.quantize(a, "e4m3", "row")
    qb = mx.quantize(b, "e4m3", "col")
    y = mx.gemm(qa, qb, "bf16")
    assert mx.device_status() == 0
    ra = O.quantize(to_f64(a[m - 64:]), "e4m3", "row")
    rb = O.quantize(to_f64(b[:, n - 256:]), "e4m3", "col")
    y_ref, t_ref = O.gemm(ra, rb)
    assert_gemm_close(y[m - 64:, n - 256:], y_ref, t_ref, "bf16")
    del a, b, qa, qb, y
    torch.cuda.empty_cache()
