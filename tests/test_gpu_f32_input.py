"""GPU parity of the quantizer on FP32 input against the oracle.

The oracle takes the FP32 values exactly (as float64), so codes and scales
must match bit for bit, including the zero padding of the swizzled scale
buffer.  An FP32 tile is 64 columns wide and fills half of each 512-byte
scale unit, so the shapes below put the last column tile in either half."""
import numpy as np
import pytest
import torch

from mxcheck import canonical_scales, ensure_built, to_f64
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu

FP8 = ["e4m3", "e5m2"]
NARROW = ["e2m3", "e3m2", "e2m1"]
PACKED = ["e2m3_packed", "e3m2_packed", "e2m1_packed"]
ALL = FP8 + NARROW + PACKED


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def special_f32(rows, cols, seed):
    """FP32 matrix mixing normal data with the block edge cases that only
    FP32 can hold: FP32 subnormals, amax significands one FP32 step above a
    format's maximum significand, values near the FP32 maximum, elements
    whose scaled value underflows FP32, and values just off the rounding
    midpoints of the element grids."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 4)
    flat = x.view(-1)
    nb = flat.numel() // 32
    kinds = torch.randint(0, 13, (nb,), generator=g)
    for b in range(nb):
        blk = flat[b * 32:(b + 1) * 32]
        k = int(kinds[b])
        e = int(torch.randint(-30, 30, (1,), generator=g))
        if k == 0:
            blk.zero_()
        elif k == 1:
            blk.zero_()
            blk[::3] = -0.0
        elif k == 2:
            blk.copy_(torch.randn(32, generator=g) * 2.0 ** -140)   # FP32 subnormals
        elif k == 3:
            blk.fill_(float(torch.randn(1, generator=g)))
        elif k == 4:
            blk.mul_(0.01)
            blk[5] = 2.0 ** e                                      # amax at a binade edge
        elif k == 5:
            # amax significand one FP32 step above 1.5, 1.75 or 1.875
            sig = (1.5, 1.75, 1.875)[int(torch.randint(0, 3, (1,), generator=g))]
            blk.mul_(0.01)
            blk[7] = (sig + 2.0 ** -22) * 2.0 ** e
        elif k == 6:
            blk.copy_(torch.randn(32, generator=g) * 1e37)
            blk[3] = 3.4028234663852886e38                           # FP32 maximum
            blk[4] = -3.4028234663852886e38
        elif k == 7:
            blk.copy_(torch.randn(32, generator=g) * 1e-37)
        elif k == 8:
            blk.copy_(torch.randn(32, generator=g) * 1e-30)        # scaled values underflow FP32
            blk[0] = 1e30
        elif k == 9:
            # 1 + j/16 +- one FP32 step: just off the E4M3 / E2M3 midpoints
            j = torch.randint(0, 16, (32,), generator=g).float()
            s = torch.randint(-1, 2, (32,), generator=g).float()
            sign = torch.randint(0, 2, (32,), generator=g).float() * 2 - 1
            blk.copy_(sign * (1 + j / 16 + s * 2.0 ** -23) * 2.0 ** e)
            blk[0] = 2.0 ** (e + 1)
    return x


def expected_codes(ref, fmt):
    if fmt in PACKED:
        return O.pack_dense(ref.codes, fmt.replace("_packed", ""))
    if fmt in NARROW:
        return O.pack_container(ref.codes, fmt)
    return ref.codes


def check(q, x, fmt, axis, rule="floor", rand=None):
    ref = O.quantize(to_f64(x), fmt.replace("_packed", ""), axis, rule, rand=rand)
    assert torch.equal(q.codes.cpu(), torch.from_numpy(expected_codes(ref, fmt))), (fmt, axis)
    assert np.array_equal(q.scales.cpu().numpy(), O.swizzle_scales(ref.scales)), (fmt, axis)
    return ref


@pytest.mark.parametrize("fmt", ALL)
@pytest.mark.parametrize("rule", ["floor", "ceil"])
@pytest.mark.parametrize("shape", [(32, 32), (96, 96), (160, 224), (416, 160), (288, 1056)])
def test_f32_quantize_matches_oracle(mx, fmt, rule, shape):
    x = special_f32(*shape, seed=shape[0] * 5 + shape[1])
    row, col = mx.quantize(x.cuda(), fmt, "both", rule)
    assert mx.device_status() == 0
    check(row, x, fmt, "row", rule)
    check(col, x, fmt, "col", rule)
    only_row = mx.quantize(x.cuda(), fmt, "row", rule)
    only_col = mx.quantize(x.cuda(), fmt, "col", rule)
    assert torch.equal(only_row.codes, row.codes) and torch.equal(only_row.scales, row.scales)
    assert torch.equal(only_col.codes, col.codes) and torch.equal(only_col.scales, col.scales)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "e3m2_packed"])
@pytest.mark.parametrize("shape", [(1, 32), (7, 96), (130, 160), (257, 1056)])
def test_f32_rowwise_ragged_rows(mx, fmt, shape):
    x = special_f32(*shape, seed=shape[0] + shape[1])
    check(mx.quantize(x.cuda(), fmt, "row"), x, fmt, "row")


@pytest.mark.parametrize("fmt", ["e5m2", "e2m3", "e2m1_packed"])
@pytest.mark.parametrize("shape", [(32, 8), (96, 200), (128, 96), (1056, 136)])
def test_f32_colwise_ragged_cols(mx, fmt, shape):
    x = special_f32(*shape, seed=shape[0] + shape[1])
    check(mx.quantize(x.cuda(), fmt, "col"), x, fmt, "col")


@pytest.mark.parametrize("fmt", ALL)
@pytest.mark.parametrize("axis", ["row", "col", "both"])
def test_f32_stochastic_rounding_matches_oracle(mx, fmt, axis):
    """Bit-exact codes given the same 16-bit random integers: with FP32
    input the fraction of a step has up to 23 bits, of which the rule reads
    the top 16."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    rows, cols = 160, 224
    x = special_f32(rows, cols, seed=77)
    rand = W.random_bits16((rows, cols), seed=78)
    got = mx.quantize(x.cuda(), fmt, axis, rand=rand.cuda())
    assert mx.device_status() == 0
    rnp = rand.numpy().view(np.uint16).astype(np.int64)
    outs = got if axis == "both" else (got,)
    axes = ("row", "col") if axis == "both" else (axis,)
    for q, ax in zip(outs, axes):
        check(q, x, fmt, ax, rand=rnp)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1_packed", "e3m2"])
def test_f32_of_bf16_values_equals_the_bf16_path(mx, fmt):
    """bf16 values widened to FP32 quantize exactly as the bf16 input does,
    in both orientations and with stochastic rounding."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    xb = W.quantize_sweep((384, 640), seed=3, device="cuda")
    rand = W.random_bits16((384, 640), seed=4, device="cuda")
    for r in (None, rand):
        a = mx.quantize(xb, fmt, "both", rand=r)
        b = mx.quantize(xb.float(), fmt, "both", rand=r)
        for qa, qb in zip(a, b):
            assert torch.equal(qa.codes, qb.codes) and torch.equal(qa.scales, qb.scales)


def test_f32_nan_and_inf_blocks(mx):
    x = special_f32(64, 192, seed=9)
    x[3, 40] = float("nan")
    x[10, 70] = float("inf")
    x[45, 130] = float("-inf")
    for fmt in ("e4m3", "e2m1"):
        row, col = mx.quantize(x.cuda(), fmt, "both")
        r = check(row, x, fmt, "row")
        c = check(col, x, fmt, "col")
        assert (r.scales == 0xFF).sum() == 3 and (c.scales == 0xFF).sum() == 3


def test_f32_strided_input(mx):
    base = special_f32(96, 324, seed=12)
    xv = base.cuda()[:, 68:260]          # ldx = 324 (16-byte rows), cols = 192
    row, col = mx.quantize(xv, "e4m3", "both")
    x = base[:, 68:260].contiguous()
    check(row, x, "e4m3", "row")
    check(col, x, "e4m3", "col")


@pytest.mark.parametrize("fmt", FP8)
def test_f32_grouped_matches_oracle(mx, fmt):
    sizes = [0, 1, 31, 200, 0, 128, 129, 5]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    total, cols = int(offsets[-1]), 224
    x = special_f32(total, cols, seed=31)
    d_off = torch.from_numpy(offsets).cuda()
    ldq = mx.mx_grouped_cols_capacity(total, len(sizes))
    row, col = mx.quantize_grouped(x.cuda(), d_off, fmt, axis="both", ldq=ldq)
    assert mx.device_status() == 0
    ref = O.quantize(to_f64(x), fmt, "row")
    assert torch.equal(row.codes.cpu(), torch.from_numpy(ref.codes))
    want = O.swizzle_scales_grouped(ref.scales, offsets)
    assert np.array_equal(row.scales.cpu().numpy()[:want.size], want)
    qs = O.quantize_grouped_cols(to_f64(x), offsets, fmt)
    codes, scales = O.pack_grouped_cols(qs, offsets, ldq)
    used = int(O.grouped_scale_rows(offsets)[-1])
    assert torch.equal(col.codes[:, :used].cpu(), torch.from_numpy(codes[:, :used]))
    got = canonical_scales(col.scales, cols, ldq)
    assert np.array_equal(got[:, :used // 32], scales[:, :used // 32])


def test_f32_quantize_16384x8192_sampled(mx):
    """Full-size FP32 launch (512 MiB in); the oracle checks sampled
    128-row / 128-column stripes (first, interior, last) of both
    orientations."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    rows, cols = 16384, 8192
    x = W.quantize_sweep((rows, cols), seed=1, device="cuda", dtype=torch.float32)
    r, c = mx.quantize(x, "e4m3", "both")
    assert mx.device_status() == 0
    rs = canonical_scales(r.scales, rows, cols)
    cs = canonical_scales(c.scales, cols, rows)
    for r0 in (0, 128 * 61, rows - 128):
        q = O.quantize(to_f64(x[r0:r0 + 128]), "e4m3", "row")
        assert torch.equal(r.codes[r0:r0 + 128].cpu(), torch.from_numpy(q.codes))
        assert np.array_equal(rs[r0:r0 + 128], q.scales)
    for c0 in (0, 64 * 61, cols - 64):
        q = O.quantize(to_f64(x[:, c0:c0 + 64]), "e4m3", "col")
        assert torch.equal(c.codes[c0:c0 + 64].cpu(), torch.from_numpy(q.codes))
        assert np.array_equal(cs[c0:c0 + 64], q.scales)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m3", "e3m2", "e2m1"])
def test_f32_ceil_rule_at_the_significand_threshold(mx, fmt):
    """Block maxima one FP32 step below, at, and one step above the
    significand of the format's maximum (1.75, 1.875 or 1.5) across
    binades: the ceil rule raises the exponent only strictly above it,
    which only the 23-bit FP32 significand can show."""
    sig = {"e4m3": 1.75, "e5m2": 1.75, "e3m2": 1.75, "e2m3": 1.875, "e2m1": 1.5}[fmt]
    rows = []
    for e in range(-20, 21, 4):
        for d in (-2.0 ** -23, 0.0, 2.0 ** -23, 2.0 ** -22):
            r = np.full(32, 0.25 * 2.0 ** e)
            r[7] = (sig + d) * 2.0 ** e
            r[9] = -(sig + d) * 2.0 ** e / 3
            rows.append(r)
    x = torch.tensor(np.array(rows), dtype=torch.float32)
    for rule in ("ceil", "floor"):
        q = mx.quantize(x.cuda(), fmt, "row", rule)
        check(q, x, fmt, "row", rule)


def test_f32_empty_quantize_writes_nothing(mx):
    """rows = 0 or cols = 0 are valid for FP32 input and launch nothing,
    also with stochastic rounding."""
    h = int(torch.cuda.current_stream().cuda_stream)
    sentinel = torch.full((256,), 0xAB, dtype=torch.uint8, device="cuda")
    x = torch.zeros(64, dtype=torch.float32, device="cuda")
    r = torch.zeros(64, dtype=torch.int16, device="cuda")
    s = sentinel.data_ptr()
    assert mx.mx_quantize(x.data_ptr(), 1, 0, 32, 32, 0, 3, 0, s, s, s, s, h) == 0
    assert mx.mx_quantize(x.data_ptr(), 1, 32, 0, 0, 0, 1, 0, s, s, None, None, h) == 0
    assert mx.mx_quantize_sr(x.data_ptr(), 1, 0, 32, 32, r.data_ptr(), 32, 1, 3, 0, s, s, s, s,
                             h) == 0
    assert mx.device_status() == 0
    assert (sentinel == 0xAB).all()


@pytest.mark.parametrize("shape,axis", [((1, 16), "row"), ((16, 8), "col"), ((16, 16), "both")])
def test_f32_smallest_shapes(mx, shape, axis):
    """The smallest legal FP32 shapes: one 16-element partial block."""
    x = special_f32(*shape, seed=shape[0] + shape[1])
    out = mx.quantize(x.cuda(), "e4m3", axis)
    assert mx.device_status() == 0
    pairs = [(out[0], "row"), (out[1], "col")] if axis == "both" else [(out, axis)]
    for q, ax in pairs:
        check(q, x, "e4m3", ax)
