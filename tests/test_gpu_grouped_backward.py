"""GPU parity of the mixture-of-experts backward pass: the grouped columnwise
quantizer (blocks inside each expert's tokens, final partial block zero
padded), the data-gradient GEMM with the experts' weights side by side
along K, and the per-expert weight-gradient GEMM grouped along K -- each
against the CPU oracle."""
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


def offsets_of(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def tokens(total, cols, seed, std=1.0, spikes=True):
    """bf16 [total, cols] N(0, std) with a few large entries (so that block
    scales differ between neighbouring blocks)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(total, cols, generator=g) * std
    if spikes and total * cols:
        idx = torch.randperm(total * cols, generator=g)[:max(1, total * cols // 500)]
        x.view(-1)[idx] *= 300.0
    return x.to(torch.bfloat16)


def check_grouped_cols(mx, q, x, offsets, fmt, ldq):
    """Codes and scales of the defined segment region against the oracle."""
    cols = x.shape[1]
    qs = O.quantize_grouped_cols(to_f64(x), offsets, fmt)
    codes, scales = O.pack_grouped_cols(qs, offsets, ldq)
    used = int(O.grouped_scale_rows(offsets)[-1])
    assert torch.equal(q.codes[:, :used].cpu(), torch.from_numpy(codes[:, :used]))
    got = canonical_scales(q.scales, cols, ldq)
    assert np.array_equal(got[:, :used // 32], scales[:, :used // 32])
    return used


GROUP_SIZES = [[0, 1, 31, 33, 0, 100, 35], [300], [128, 128], [0, 0, 5], [1] * 9,
               [64, 0, 257, 0]]


@pytest.mark.parametrize("sizes", GROUP_SIZES)
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_grouped_cols_quantize_matches_oracle(mx, sizes, fmt):
    offsets = offsets_of(sizes)
    total = int(offsets[-1])
    x = tokens(total, 200, seed=total + len(sizes))
    d_off = torch.from_numpy(offsets).cuda()
    ldq = mx.mx_grouped_cols_capacity(total, len(sizes))
    q = mx.quantize_grouped(x.cuda(), d_off, fmt, axis="col", ldq=ldq)
    assert mx.device_status() == 0
    assert q.codes.shape == (200, ldq)
    check_grouped_cols(mx, q, x, offsets, fmt, ldq)


def test_grouped_both_from_one_read(mx):
    sizes = [0, 1, 31, 33, 0, 100, 35]
    offsets = offsets_of(sizes)
    total = int(offsets[-1])
    x = tokens(total, 256, seed=3).cuda()
    d_off = torch.from_numpy(offsets).cuda()
    row, col = mx.quantize_grouped(x, d_off, "e4m3", axis="both", ldq=1024)
    row_only = mx.quantize_grouped(x, d_off, "e4m3")
    col_only = mx.quantize_grouped(x, d_off, "e4m3", axis="col", ldq=1024)
    assert mx.device_status() == 0
    assert torch.equal(row.codes, row_only.codes)
    assert torch.equal(row.scales, row_only.scales)
    assert torch.equal(col.codes, col_only.codes)
    assert torch.equal(col.scales, col_only.scales)
    check_grouped_cols(mx, col, x.cpu(), offsets, "e4m3", 1024)


def test_grouped_cols_leave_the_tail_untouched_and_reject_overflow(mx):
    """Columns past the last group are not written; a layout that does not
    fit in ldq is reported on the device and nothing is written."""
    sizes = [100, 0, 30]
    offsets = offsets_of(sizes)
    x = tokens(130, 64, seed=5).cuda()
    d_off = torch.from_numpy(offsets).cuda()
    h = int(torch.cuda.current_stream().cuda_stream)
    for ldq, status in ((512, 0), (128, 6)):
        q = torch.full((64, ldq), 0xAB, dtype=torch.uint8, device="cuda")
        s = torch.full((mx.mx_scale_bytes(64, ldq),), 0xCD, dtype=torch.uint8, device="cuda")
        st = mx.mx_quantize_grouped_ex(x.data_ptr(), 0, 130, 64, 64, 0, 2, 0, 3, d_off.data_ptr(),
                                       None, None, q.data_ptr(), ldq, s.data_ptr(), h)
        assert st == 0
        assert mx.device_status() == status
        if status == 0:
            assert (q[:, 256:] == 0xAB).all()           # two 128-column segments used
            assert (q[:, 100:128] == 0).all()           # padding tokens are code 0
        else:
            assert (q == 0xAB).all() and (s == 0xCD).all()


def run_dgrad(mx, sizes, n_model, n_expert, out, seed=0):
    """dX_g = dY_g W_g^T with W stored [E, n_expert, n_model] (each expert's
    W^T): dY rowwise E5M2 (blocks along n_expert), the stacked weights
    quantized columnwise once ([n_model, E*n_expert])."""
    offsets = offsets_of(sizes)
    groups, total = len(sizes), int(offsets[-1])
    dy = tokens(total, n_expert, seed, std=1e-3)
    g = torch.Generator().manual_seed(seed + 1)
    w = (torch.randn(groups, n_expert, n_model, generator=g) * 0.02).to(torch.bfloat16)
    d_off = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(dy.cuda(), d_off, "e5m2")
    qb = mx.quantize(w.cuda().view(groups * n_expert, n_model), "e4m3", "col")
    tdtype = torch.float32 if out == "fp32" else torch.bfloat16
    buf = torch.full((total + 8, n_model), float("nan"), dtype=tdtype, device="cuda")
    y = mx.grouped_gemm_bcat(qa, d_off, qb, out, out=buf[:total])
    assert mx.device_status() == 0
    assert torch.isnan(buf[total:].float()).all()
    a = O.quantize(to_f64(dy), "e5m2", "row")
    bs = [O.quantize(to_f64(w[e]), "e4m3", "col") for e in range(groups)]
    assert torch.equal(qb.codes.cpu(), torch.from_numpy(np.concatenate([b.codes for b in bs], 1)))
    y_ref, t_ref = O.grouped_gemm(a, offsets, bs)
    assert_gemm_close(y, y_ref, t_ref, out)


@pytest.mark.parametrize("sizes", [[0, 1, 31, 200, 0, 128, 129, 5], [300], [0, 0, 77]])
def test_grouped_dgrad_bcat_matches_oracle(mx, sizes):
    run_dgrad(mx, sizes, 264, 256, "fp32", seed=len(sizes))


def test_grouped_dgrad_bcat_bf16_long_k(mx):
    run_dgrad(mx, [3, 0, 250, 64], 384, 1152, "bf16", seed=11)


def run_wgrad(mx, sizes, m, n, out, seed=0, ldq=None):
    """dW_g = dY_g^T X_g over each expert's tokens: both operands from the
    grouped columnwise quantizer."""
    offsets = offsets_of(sizes)
    groups, total = len(sizes), int(offsets[-1])
    dy = tokens(total, m, seed, std=1e-3)
    x = tokens(total, n, seed + 1)
    d_off = torch.from_numpy(offsets).cuda()
    ldq = ldq or mx.mx_grouped_cols_capacity(total, groups)
    qa = mx.quantize_grouped(dy.cuda(), d_off, "e5m2", axis="col", ldq=ldq)
    qb = mx.quantize_grouped(x.cuda(), d_off, "e4m3", axis="col", ldq=ldq)
    y = mx.grouped_gemm_wgrad(qa, d_off, qb, total, out)
    assert mx.device_status() == 0
    assert y.shape == (groups, m, n)
    check_grouped_cols(mx, qa, dy, offsets, "e5m2", ldq)
    check_grouped_cols(mx, qb, x, offsets, "e4m3", ldq)
    a = O.quantize_grouped_cols(to_f64(dy), offsets, "e5m2")
    b = O.quantize_grouped_cols(to_f64(x), offsets, "e4m3")
    y_ref, t_ref = O.grouped_wgrad(a, b)
    for e in range(groups):
        if sizes[e] == 0:
            assert int((y[e] != 0).sum()) == 0, "an expert without tokens must get zeros"
    assert_gemm_close(y, y_ref, t_ref, out)


@pytest.mark.parametrize("sizes", [[0, 1, 31, 33, 0, 100, 35], [300], [0, 0, 77], [1] * 9,
                                   [129, 0, 640]])
def test_grouped_wgrad_matches_oracle(mx, sizes):
    run_wgrad(mx, sizes, 256, 264, "fp32", seed=len(sizes))


@pytest.mark.parametrize("sizes", [[1000, 0, 37, 2000, 5, 800, 64], [900, 1], [3000]])
def test_grouped_wgrad_long_and_short_experts(mx, sizes):
    """Experts with many tokens (long contractions over many K stages)
    beside experts with a few tokens or none, with several m- and n-tiles
    per expert."""
    run_wgrad(mx, sizes, 512, 520, "fp32", seed=sum(sizes) % 97)


def test_grouped_wgrad_is_deterministic(mx):
    """Repeated calls agree bit for bit (each output tile's contraction
    order is fixed)."""
    sizes = [1500, 3, 0, 700, 41, 2100, 9]
    offsets = offsets_of(sizes)
    total = int(offsets[-1])
    dy = tokens(total, 768, 5, std=1e-3).cuda()
    x = tokens(total, 512, 6).cuda()
    d_off = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(dy, d_off, "e5m2", axis="col")
    qb = mx.quantize_grouped(x, d_off, "e4m3", axis="col")
    first = mx.grouped_gemm_wgrad(qa, d_off, qb, total, "fp32")
    for _ in range(3):
        assert torch.equal(first, mx.grouped_gemm_wgrad(qa, d_off, qb, total, "fp32"))
    assert mx.device_status() == 0


def test_grouped_wgrad_bf16_and_ragged_m(mx):
    run_wgrad(mx, [5, 0, 300, 40], 328, 128, "bf16", seed=13)


def test_grouped_wgrad_rejects_bad_offsets_and_overflow(mx):
    sizes = [40, 60]
    offsets = offsets_of(sizes)
    dy = tokens(100, 128, 1, std=1e-3).cuda()
    x = tokens(100, 128, 2).cuda()
    good = torch.from_numpy(offsets).cuda()
    qa = mx.quantize_grouped(dy, good, "e5m2", axis="col", ldq=256)
    qb = mx.quantize_grouped(x, good, "e4m3", axis="col", ldq=256)
    assert mx.device_status() == 0
    y = torch.zeros(2, 128, 128, device="cuda")
    for bad in ([0, 70, 60], [1, 40, 100], [0, 40, 99]):
        mx.grouped_gemm_wgrad(qa, torch.tensor(bad, dtype=torch.int32, device="cuda"), qb, 100,
                              out=y)
        assert mx.device_status() == 6
        assert int(y.abs().sum()) == 0
    # segments that do not fit in the operands' 128 columns
    small = mx.MxTensor(qa.codes[:, :128].contiguous(), qa.scales, "e5m2")
    smallb = mx.MxTensor(qb.codes[:, :128].contiguous(), qb.scales, "e4m3")
    mx.grouped_gemm_wgrad(small, good, smallb, 100, out=y)
    assert mx.device_status() == 6
    assert int(y.abs().sum()) == 0
    mx.grouped_gemm_wgrad(qa, good, qb, 100, out=y)
    assert mx.device_status() == 0
    assert int(y.abs().sum()) > 0


def test_moe_backward_full_size_sampled(mx):
    """64 experts, K = 7168, N = 2048, 65 536 routed tokens (Zipf split with
    empty and sub-32-row groups): dgrad and wgrad at full size, every
    expert checked on sampled rows and columns against the oracle."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    x, w, offsets = W.moe_inputs(device="cuda")
    experts, n, k = w.shape
    dy = W.moe_grad_output(device="cuda")
    total = x.shape[0]
    d_off = torch.from_numpy(offsets).cuda()
    sizes = np.diff(offsets)
    rng = np.random.default_rng(1)

    # data gradient: dX [total, k] = per expert dY_g [m_g, n] * W_g [n, k]
    qa = mx.quantize_grouped(dy, d_off, "e5m2")
    qb = mx.quantize(w.view(experts * n, k), "e4m3", "col")
    dx = mx.grouped_gemm_bcat(qa, d_off, qb, "fp32")
    assert mx.device_status() == 0
    kcols = np.unique(np.concatenate([np.arange(0, 32), rng.choice(k, 32, replace=False),
                                      np.arange(k - 32, k)]))
    kcols_t = torch.from_numpy(kcols).cuda()
    for e in range(experts):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        rows = np.unique(np.concatenate([np.arange(lo, min(hi, lo + 3)),
                                         np.arange(max(lo, hi - 3), hi)]))
        rows_t = torch.from_numpy(rows).cuda()
        ra = O.quantize(to_f64(dy[rows_t]), "e5m2", "row")
        bq = O.quantize(to_f64(w[e][:, kcols_t]), "e4m3", "col")       # [len(kcols), n]
        assert torch.equal(qb.codes[kcols_t][:, e * n:(e + 1) * n].cpu(), torch.from_numpy(bq.codes))
        y_ref, t_ref = O.gemm(ra, bq)
        assert_gemm_close(dx[rows_t][:, kcols_t], y_ref, t_ref, "fp32")
    del dx, qa, qb

    # weight gradient: dW [experts, n, k], dW_g = dY_g^T X_g
    ldq = mx.mx_grouped_cols_capacity(total, experts)
    qa = mx.quantize_grouped(dy, d_off, "e5m2", axis="col", ldq=ldq)
    qb = mx.quantize_grouped(x, d_off, "e4m3", axis="col", ldq=ldq)
    dw = mx.grouped_gemm_wgrad(qa, d_off, qb, total, "fp32")
    assert mx.device_status() == 0
    ncols = np.unique(np.concatenate([[0, 1, n - 1], rng.choice(n, 8, replace=False)]))
    ncols_t = torch.from_numpy(ncols).cuda()
    for e in range(experts):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            assert int((dw[e] != 0).sum()) == 0
            continue
        sub_off = [0, hi - lo]
        a = O.quantize_grouped_cols(to_f64(dy[lo:hi][:, ncols_t]), sub_off, "e5m2")
        b = O.quantize_grouped_cols(to_f64(x[lo:hi][:, kcols_t]), sub_off, "e4m3")
        y_ref, t_ref = O.grouped_wgrad(a, b)
        assert_gemm_close(dw[e][ncols_t][:, kcols_t], y_ref[0], t_ref[0], "fp32")
    assert (sizes == 0).sum() >= 2


def test_grouped_backward_largest_group_count(mx):
    """1000 experts (the library's maximum), most of them without tokens and
    a few ragged: the data gradient (experts side by side along K) and the
    weight gradient (grouped along K, zeros for the empty experts) read
    every entry of the device group table."""
    sizes = np.zeros(1000, dtype=np.int64)
    rng = np.random.default_rng(21)
    sizes[rng.choice(1000, 10, replace=False)] = rng.integers(1, 300, 10)
    sizes = [int(v) for v in sizes]
    run_dgrad(mx, sizes, 136, 128, "fp32", seed=21)
    run_wgrad(mx, sizes, 128, 136, "fp32", seed=22)
