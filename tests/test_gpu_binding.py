"""The tensor API's checks: every GEMM wrapper rejects, before anything is
launched, tensors whose dtype, shape, strides or byte counts do not match
what the kernels will read and write (the C ABI sees only raw pointers)."""
import pytest
import torch

from mxcheck import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def operands(mx, m=256, n=256, k=256):
    g = torch.Generator().manual_seed(3)
    x = torch.randn(m, k, generator=g).to(torch.bfloat16).cuda()
    w = torch.randn(k, n, generator=g).to(torch.bfloat16).cuda()
    return mx.quantize(x, "e4m3", "row"), mx.quantize(w, "e4m3", "col")


def test_gemm_rejects_mismatched_tensors(mx):
    qa, qb = operands(mx)
    y = mx.gemm(qa, qb, "fp32")
    assert mx.device_status() == 0
    sentinel = y.clone()
    with pytest.raises(ValueError):       # wrong output dtype
        mx.gemm(qa, qb, "bf16", out=y)
    with pytest.raises(ValueError):       # wrong output shape
        mx.gemm(qa, qb, "fp32", out=y[:128])
    with pytest.raises(ValueError):       # transposed output
        mx.gemm(qa, qb, "fp32", out=torch.empty(256, 256, device="cuda").t())
    short = mx.MxTensor(qa.codes, qa.scales[:100], "e4m3")
    with pytest.raises(ValueError):       # scales shorter than the operand needs
        mx.gemm(short, qb, "fp32", out=y)
    strided = mx.MxTensor(torch.empty(256, 512, dtype=torch.uint8, device="cuda")[:, :256],
                          qa.scales, "e4m3")
    with pytest.raises(ValueError):       # non-contiguous codes
        mx.gemm(strided, qb, "fp32", out=y)
    with pytest.raises(ValueError):       # codes of the wrong dtype
        mx.gemm(mx.MxTensor(qa.codes.view(torch.int8), qa.scales, "e4m3"), qb, "fp32", out=y)
    torch.cuda.synchronize()
    assert torch.equal(y, sentinel)       # nothing was written
    assert mx.device_status() == 0


def test_grouped_wrappers_reject_mismatched_tensors(mx):
    groups, n, k, total = 2, 128, 128, 200
    g = torch.Generator().manual_seed(4)
    x = torch.randn(total, k, generator=g).to(torch.bfloat16).cuda()
    w = torch.randn(groups * n, k, generator=g).to(torch.bfloat16).cuda()
    off = torch.tensor([0, 120, 200], dtype=torch.int32, device="cuda")
    qa = mx.quantize_grouped(x, off, "e4m3")
    qw = mx.quantize(w, "e4m3", "row")
    qb = mx.MxTensor(qw.codes.view(groups, n, k), qw.scales, "e4m3")
    y = mx.grouped_gemm(qa, off, qb, "fp32")
    assert mx.device_status() == 0
    with pytest.raises(ValueError):       # offsets of the wrong dtype
        mx.grouped_gemm(qa, off.long(), qb, "fp32", out=y)
    with pytest.raises(ValueError):       # offsets for another group count
        mx.grouped_gemm(qa, off[:2], qb, "fp32", out=y)
    with pytest.raises(ValueError):       # grouped outputs have no leading dimension: contiguous only
        mx.grouped_gemm(qa, off, qb, "fp32",
                        out=torch.empty(total, 2 * n, device="cuda")[:, :n])
    with pytest.raises(ValueError):       # expert scales shorter than groups x one matrix
        mx.grouped_gemm(qa, off, mx.MxTensor(qb.codes, qb.scales[:512], "e4m3"), "fp32", out=y)
    # weight gradient: [groups, m, n] contiguous output
    ldq = mx.mx_grouped_cols_capacity(total, groups)
    ca = mx.quantize_grouped(x, off, "e4m3", axis="col", ldq=ldq)
    cb = mx.quantize_grouped(x, off, "e4m3", axis="col", ldq=ldq)
    with pytest.raises(ValueError):
        mx.grouped_gemm_wgrad(ca, off, cb, total, "fp32", out=torch.empty(groups, k, k + 8,
                                                                          device="cuda"))
    dw = mx.grouped_gemm_wgrad(ca, off, cb, total, "fp32")
    assert dw.shape == (groups, k, k)
    assert mx.device_status() == 0
