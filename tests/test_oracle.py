"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/*.json, each with its citation), an independent
library routine (torch's float8 dtypes), exact rational arithmetic, brute
force, or a closed form.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


# ---------------------------------------------------------------- decoding

@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_decode_all_codes_match_torch(fmt):
    """All 256 codes decode like torch's OCP float8 dtype (library routine)."""
    mine = O.decode_table(fmt)
    ref = torch.arange(256, dtype=torch.uint8).view(TORCH_FP8[fmt]).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))


def test_format_facts_from_page(golden_dir):
    g = load(golden_dir, "format_facts.json")
    t4 = O.decode_table("e4m3")
    e4 = g["e4m3"]
    finite = t4[np.isfinite(t4)]
    assert finite.max() == e4["max"] and t4[0x7E] == 448.0 and t4[0xFE] == -448.0
    assert [c for c in range(256) if np.isnan(t4[c])] == e4["nan_codes"]
    assert not np.isinf(t4).any()
    pos = np.sort(finite[finite > 0])
    assert pos[0] == e4["min_subnormal"]
    assert pos[pos >= e4["min_normal"]][0] == e4["min_normal"]
    assert pos[pos < e4["min_normal"]].max() < e4["min_normal"]
    for lo, hi, step in e4["spacing"]:
        grid = pos[(pos >= lo) & (pos <= hi)]
        assert np.all(np.diff(grid) == step)
    t5 = O.decode_table("e5m2")
    f5 = t5[np.isfinite(t5)]
    assert f5.max() == g["e5m2"]["max"]
    assert np.sort(f5[f5 > 0])[0] == g["e5m2"]["min_subnormal"]
    pos5 = np.sort(f5[f5 > 0])
    for lo, hi, step in g["e5m2"]["spacing"]:
        grid = pos5[(pos5 >= lo) & (pos5 < hi)]
        assert np.all(np.diff(grid) == step)
    assert np.isinf(t5).sum() == 2


def test_e8m0_decode_from_page(golden_dir):
    g = load(golden_dir, "e8m0.json")
    for code, val in g["decode"].items():
        assert O.decode_e8m0(int(code)) == val
    assert O.decode_e8m0(0) > 0
    assert math.isnan(O.decode_e8m0(g["nan_code"]))
    with pytest.raises(ValueError):
        O.decode_e8m0(256)
    vals = O.e8m0_values(np.array([0x77, 0x80, 0, 255], dtype=np.uint8))
    assert vals[0] == 2.0 ** -8 and vals[1] == 2.0 and vals[2] == 2.0 ** -127
    assert math.isnan(vals[3])


def test_payload_model_from_page(golden_dir):
    """Two rows of 32 E4M3 codes: 64 code bytes + 4 (FP32 tensor scale) = 68,
    or + 2 E8M0 block scales = 66; the scale overheads are 6.25% / 3.125%."""
    g = load(golden_dir, "e8m0.json")
    codes = 2 * O.BLOCK
    assert codes + 4 == g["payload_bytes"]["two_rows_of_32_e4m3_tensor_scale"]
    assert codes + 2 * 1 == g["payload_bytes"]["two_rows_of_32_e4m3_mx"]
    assert 100 * 4 / codes == g["scale_overhead_percent"]["tensor"]
    assert 100 * 2 / codes == g["scale_overhead_percent"]["mx"]


# ---------------------------------------------------------------- encoding

def test_cast_audit_from_page(golden_dir):
    g = load(golden_dir, "cast_audit.json")
    codes = O.encode_sat_rne(g["fmt"], np.array(g["inputs"]))
    vals = O.decode_table(g["fmt"])[codes]
    assert vals.tolist() == g["outputs"]
    assert np.signbit(vals).tolist() == g["output_signbit"]
    t = O.decode_table("e4m3")
    for code, val in g["byte_decoding"].items():
        assert t[int(code, 16)] == val and np.signbit(t[int(code, 16)]) == np.signbit(val)


def test_saturation_and_rne_from_page(golden_dir):
    g = load(golden_dir, "format_facts.json")
    t4 = O.decode_table("e4m3")
    for x, y in g["e4m3"]["saturate"]:
        assert t4[O.encode_sat_rne("e4m3", np.array([x]))[0]] == y
        assert t4[O.encode_sat_rne("e4m3", np.array([-x]))[0]] == -y
    r = g["rounding"]
    assert t4[O.encode_sat_rne(r["fmt"], np.array([r["x"]]))[0]] == r["rne"]
    lo, hi = r["neighbors"]
    grid = np.sort(t4[np.isfinite(t4)])
    assert lo in grid and hi in grid and not np.any((grid > lo) & (grid < hi))
    t5 = O.decode_table("e5m2")
    for x in [57344.0, 60000.0, 61440.0, 1e9, math.inf]:
        assert t5[O.encode_sat_rne("e5m2", np.array([x]))[0]] == 57344.0
    assert O.encode_sat_rne("e4m3", np.array([math.inf]))[0] == 0x7E
    assert O.encode_sat_rne("e4m3", np.array([math.nan]))[0] == O.NAN_CODE


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_every_bf16_pattern_matches_torch(fmt):
    """Exhaustive: every finite bf16 value, scale 1, against torch's RNE cast
    of the value pre-clamped to the finite range (an independent routine)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_bits_to_float64(bits)
    ok = np.isfinite(vals)
    vals = vals[ok]
    mine = O.encode_sat_rne(fmt, vals)
    mx = O.FORMATS[fmt].max_finite
    ref = torch.from_numpy(np.clip(vals, -mx, mx)).float().to(TORCH_FP8[fmt])
    ref = ref.view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_decode_round_trip(fmt):
    t = O.decode_table(fmt)
    codes = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    assert np.array_equal(O.encode_sat_rne(fmt, t[codes]), codes)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_midpoints_tie_to_even_code(fmt):
    """Between adjacent positive finite codes c, c+1 (consecutive integers),
    the exact midpoint goes to the one with an even mantissa LSB, slightly
    off the midpoint goes to the nearer one."""
    t = O.decode_table(fmt)
    for c in range(0, 0x7F):
        lo, hi = t[c], t[c + 1]
        if not (np.isfinite(lo) and np.isfinite(hi)):
            continue
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert O.encode_sat_rne(fmt, np.array([mid]))[0] == even
        assert O.encode_sat_rne(fmt, np.array([-mid]))[0] == even | 0x80
        eps = (hi - lo) / 1024
        assert O.encode_sat_rne(fmt, np.array([mid - eps]))[0] == c
        assert O.encode_sat_rne(fmt, np.array([mid + eps]))[0] == c + 1


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_is_monotone_and_keeps_sign(fmt):
    rng = np.random.default_rng(5)
    v = np.sort(np.concatenate([rng.standard_normal(20000) * s for s in (1e-4, 1, 100, 1e5)]))
    vals = O.decode_table(fmt)[O.encode_sat_rne(fmt, v)]
    assert np.all(np.diff(vals) >= 0)
    assert np.all(np.signbit(vals) == np.signbit(v))


# ---------------------------------------------------------------- block scales

def test_floor_rule_puts_scaled_amax_in_top_binade():
    """OCP floor rule: after scaling, amax lies in [2^emax, 2^(emax+1))."""
    rng = np.random.default_rng(1)
    amax = np.exp(rng.uniform(-60, 60, 5000))  # no exponent clamping here
    for fmt in ("e4m3", "e5m2"):
        f = O.FORMATS[fmt]
        e = O.scale_exponent_floor(fmt, amax)
        s = amax * 2.0 ** (-e.astype(np.float64))
        assert np.all((s >= 2.0 ** f.emax_elem) & (s < 2.0 ** (f.emax_elem + 1)))


def test_ceil_rule_brute_force():
    """Page's conservative rule: the smallest e in [-127, 200] with
    amax <= max * 2^e, found by linear search with exact comparisons."""
    rng = np.random.default_rng(2)
    amax = np.concatenate([np.exp(rng.uniform(-60, 60, 300)),
                           [448.0, 449.0, 447.0, 896.0, 2.0 ** -140, 57344.0]])
    for fmt in ("e4m3", "e5m2"):
        mx = O.FORMATS[fmt].max_finite
        got = O.scale_exponent_ceil(fmt, amax)
        for a, e in zip(amax, got):
            want = next(k for k in range(-127, 200) if a <= mx * 2.0 ** k)
            assert e == want


def test_ceil_equals_floor_plus_one_iff_significand_above_1_75():
    rng = np.random.default_rng(3)
    amax = np.exp(rng.uniform(-40, 40, 20000))
    sig = amax / 2.0 ** O.floor_log2_exact(amax)
    for fmt in ("e4m3", "e5m2"):
        diff = O.scale_exponent_ceil(fmt, amax) - O.scale_exponent_floor(fmt, amax)
        assert np.array_equal(diff, (sig > 1.75).astype(np.int64))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantize_codes_match_torch_cast_given_scale(fmt):
    """Given each block's scale, the codes equal torch's RNE cast of the
    exactly scaled, pre-clamped values."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-10, 10, (64, 1)))
    x[rng.random(x.shape) < 0.01] *= 300
    x = O.bf16_bits_to_float64((x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    q = O.quantize(x, fmt, "row")
    s = O.e8m0_values(q.scales)
    scaled = x.reshape(64, 8, 32) / s[:, :, None]
    mx = O.FORMATS[fmt].max_finite
    ref = torch.from_numpy(np.clip(scaled, -mx, mx).reshape(64, 256)).float()
    ref = ref.to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(q.codes, ref)


def test_zero_nan_inf_and_subnormal_blocks():
    x = np.zeros((4, 64))
    x[0, 5] = -0.0
    x[1, :32] = np.nan
    x[1, 40] = 1.0
    x[2, 3] = np.inf
    x[3, :32] = 2.0 ** -133          # smallest bf16 subnormal
    x[3, 32:] = 3 * 2.0 ** -130
    q = O.quantize(x, "e4m3", "row")
    assert q.scales[0].tolist() == [127, 127]          # zero block: S = 1
    assert q.codes[0, 5] == 0x80 and q.codes[0, 4] == 0
    assert q.scales[1].tolist() == [255, 127 - 8]
    assert np.all(q.codes[1, :32] == O.NAN_CODE)
    assert q.scales[2, 0] == 255 and np.all(q.codes[2, :32] == O.NAN_CODE)
    assert q.scales[3].tolist() == [0, 0]               # clamped at 2^-127
    t = O.decode_table("e4m3")
    assert t[q.codes[3, 0]] == 2.0 ** -6 and t[q.codes[3, 32]] == 3 * 2.0 ** -3
    assert np.isnan(O.dequantize(q)[1, :32]).all()


def test_column_blocks_run_along_rows():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((64, 48))
    x[3, 7] = 1000.0
    qc = O.quantize(x, "e4m3", "col")
    assert qc.codes.shape == (48, 64) and qc.scales.shape == (48, 2)
    qr = O.quantize(x.T.copy(), "e4m3", "row")
    assert np.array_equal(qc.codes, qr.codes) and np.array_equal(qc.scales, qr.scales)
    big = qc.scales[7, 0]
    assert big > qc.scales[7, 1] and big > qc.scales[6, 0] and big > qc.scales[8, 0]


# ---------------------------------------------------------------- two-row experiment

def two_row_fixture(g):
    x = np.array([g["pattern_small"] * g["repeat"], g["pattern_large"] * g["repeat"]],
                 dtype=np.float32).astype(np.float64)
    w = np.array(g["weight_pattern"] * g["repeat"], dtype=np.float32).astype(np.float64)
    return x, w.reshape(32, 1)


def test_two_row_experiment_ceil_rule_from_page(golden_dir):
    g = load(golden_dir, "two_row_fixture.json")
    c = g["ceil_rule"]
    x, w = two_row_fixture(g)
    qx = O.quantize(x, "e4m3", "row", rule="ceil")
    qw = O.quantize(w, "e4m3", "col", rule="ceil")
    assert [O.decode_e8m0(int(s)) for s in qx.scales[:, 0]] == c["x_scales"]
    xh = O.dequantize(qx)
    assert round(xh[0, 0], 8) == c["x_hat_0_0"]
    assert xh[1, 3] == c["x_hat_1_3"]
    y, _ = O.gemm(qx, qw)
    d = c["print_decimals"]
    assert [round(v, d) for v in y.ravel()] == c["mx_y"]
    ref = (x @ w).ravel()
    ref32 = (x.astype(np.float32) @ w.astype(np.float32)).ravel()  # the page's FP32 matmul
    assert [round(float(v), d) for v in ref32] == c["reference_y"]
    err = np.abs(y.ravel() - ref)
    assert abs(err[0] - c["mx_abs_error"][0]) < 1e-7 and err[1] == c["mx_abs_error"][1]
    sel = np.zeros((32, 1))
    sel[3, 0] = 1.0
    ys, _ = O.gemm(qx, O.quantize(sel, "e4m3", "col", rule="ceil"))
    assert ys.ravel().tolist() == c["selector_mx"]
    assert (x @ sel).ravel().tolist() == c["selector_reference"]


def test_two_row_experiment_tensor_scale_from_page(golden_dir):
    """The tensor-wide column: one FP32 scale amax/448 for all of X."""
    g = load(golden_dir, "two_row_fixture.json")
    ts = g["tensor_scale"]
    x, w = two_row_fixture(g)
    sx = np.float32(np.abs(x).max()) / np.float32(448.0)
    sw = np.float32(np.abs(w).max()) / np.float32(448.0)
    assert round(float(sx), 6) == ts["tensor_scale_x"]
    xq = O.decode_table("e4m3")[O.encode_sat_rne("e4m3", x / float(sx))] * float(sx)
    wq = O.decode_table("e4m3")[O.encode_sat_rne("e4m3", w / float(sw))] * float(sw)
    assert xq[0, 0] == ts["x_hat_0_0"]
    y = (xq.astype(np.float32) @ wq.astype(np.float32)).ravel()  # the page's FP32 matmul
    assert [round(float(v), 6) for v in y] == ts["tensor_y"]


def test_two_row_experiment_floor_rule_saturates_spike(golden_dir):
    """Floor rule on the same fixture: the spike row's scale is 2^0, so 500
    saturates to 448 (derived from the rule; not printed by the page)."""
    g = load(golden_dir, "two_row_fixture.json")
    x, w = two_row_fixture(g)
    qx = O.quantize(x, "e4m3", "row")
    assert [O.decode_e8m0(int(s)) for s in qx.scales[:, 0]] == [2.0 ** -8, 1.0]
    assert O.dequantize(qx)[1, 3] == 448.0 and qx.codes[1, 3] == 0x7E
    y, _ = O.gemm(qx, O.quantize(w, "e4m3", "col"))
    assert y.ravel().tolist() == [0.6015625, 23.75]


# The three changes to the two-row fixture proposed in "Troubleshooting
# numerical failures" (same page).  The page prints no numbers for them;
# every expected value below is derived by hand from the format grid and
# the two scale rules, not by the oracle.
#  (1) the small row all zeros;
#  (2) 500 moved into the small row's (only) 32-value group: the reading
#      taken is x[0, 3] := 500, replacing the 0.5 at the column where the
#      spike sits in the large row; the large row is left as it is;
#  (3) W replaced by a column that selects only the spike (column 3).

def selector_w():
    sel = np.zeros((32, 1))
    sel[3, 0] = 1.0
    return sel


@pytest.mark.parametrize("rule", ["ceil", "floor"])
def test_troubleshooting_zero_small_row(golden_dir, rule):
    g = load(golden_dir, "two_row_fixture.json")
    x, w = two_row_fixture(g)
    x[0, :] = 0.0
    qx = O.quantize(x, "e4m3", "row", rule=rule)
    # an all-zero block takes S = 1 (byte 127) and every code is +0
    assert qx.scales[0, 0] == 127 and not qx.codes[0].any()
    # the spike row keeps its scale: 2 (ceil) or 1 (floor)
    assert O.decode_e8m0(int(qx.scales[1, 0])) == (2.0 if rule == "ceil" else 1.0)
    y, t = O.gemm(qx, O.quantize(w, "e4m3", "col", rule=rule))
    # nothing to lose in row 0: its projection is exactly 0
    assert y[0, 0] == 0.0 and t[0, 0] == 0.0
    assert y[1, 0] == (7.75 if rule == "ceil" else 23.75)


# Reconstructed small row (one period of the 8-value pattern) after 500
# joins its block, worked out by hand:
#  ceil rule: S = 2^ceil(log2(500/448)) = 2; 0.001/2 = 0.0005 is below half
#    the smallest subnormal 2^-9, so it becomes 0; 0.03/2 = 0.015 rounds to
#    2^-6 (8 subnormal steps of 2^-9); 0.117/2 = 0.0585 rounds to 15 * 2^-8;
#    500/2 = 250 rounds to 256 (spacing 16 in [128, 256)); the rest are
#    exact multiples of their spacing.
#  floor rule: S = 2^(floor(log2 500) - 8) = 1; 0.001 is above 2^-10, so it
#    becomes 2^-9; 0.03 rounds to 15 * 2^-9; 0.117 to 15 * 2^-7; 500
#    saturates to 448.
SPIKED_SMALL_ROW = {
    "ceil": (2.0, [0.0, 2 * 2.0 ** -6, 2 * 15 * 2.0 ** -8, 512.0,
                   1.0, -0.25, 0.0625, -0.015625]),
    "floor": (1.0, [2.0 ** -9, 15 * 2.0 ** -9, 15 * 2.0 ** -7, 448.0,
                    1.0, -0.25, 0.0625, -0.015625]),
}


@pytest.mark.parametrize("rule", ["ceil", "floor"])
def test_troubleshooting_spike_moved_into_small_row(golden_dir, rule):
    g = load(golden_dir, "two_row_fixture.json")
    x, w = two_row_fixture(g)
    x[0, 3] = 500.0
    qx = O.quantize(x, "e4m3", "row", rule=rule)
    scale, period = SPIKED_SMALL_ROW[rule]
    assert O.decode_e8m0(int(qx.scales[0, 0])) == scale
    xh = O.dequantize(qx)
    assert xh[0, :8].tolist() == period
    # columns 11, 19, 27 still hold the pattern's 0.5 (exact under either scale)
    assert xh[0, 8:].tolist() == (period[:3] + [0.5] + period[4:]) * 3
    # the page's lesson: 0.001 shares a scale with 500 and loses its precision
    # (original fixture, ceil rule: 0.00097656, 2.3 % off)
    assert abs(xh[0, 0] - 0.001) / 0.001 > 0.9
    # the large row is untouched
    assert np.array_equal(qx.codes[1], O.quantize(two_row_fixture(g)[0], "e4m3", "row",
                                                   rule=rule).codes[1])
    # the selector exposes the spike's reconstruction in both rows
    ys, _ = O.gemm(qx, O.quantize(selector_w(), "e4m3", "col", rule=rule))
    spike = 512.0 if rule == "ceil" else 448.0
    assert ys.ravel().tolist() == [spike, spike]


# Incident-trace counts for the two-row fixture and the page's troubleshooting
# changes, derived by hand: (clip count, zero count).  Original fixture: the
# ceil rule never clips (amax <= 448 S by construction) and keeps every small
# value non-zero (S = 2^-8); the floor rule keeps S = 1 for the large row, so
# its four 500s (500 > 448) are clipped.  500 moved into the small row's
# block: under the ceil rule S = 2 and the four 0.001s (0.0005 after scaling,
# below half the smallest subnormal 2^-9) become zeros; under the floor rule
# S = 1 keeps them (2^-9) and the moved 500 is clipped beside the large
# row's four.  An all-zero small row has no non-zero value to lose.
INCIDENT_COUNTS = {
    ("original", "ceil"): (0, 0), ("original", "floor"): (4, 0),
    ("spike", "ceil"): (0, 4), ("spike", "floor"): (5, 0),
    ("zero_row", "ceil"): (0, 0), ("zero_row", "floor"): (4, 0),
}


@pytest.mark.parametrize("variant", ["original", "spike", "zero_row"])
@pytest.mark.parametrize("rule", ["ceil", "floor"])
def test_incident_trace_counts_on_the_fixture(golden_dir, variant, rule):
    g = load(golden_dir, "two_row_fixture.json")
    x, _ = two_row_fixture(g)
    if variant == "spike":
        x[0, 3] = 500.0
    elif variant == "zero_row":
        x[0, :] = 0.0
    t = O.incident_trace(x, "e4m3", "row", rule)
    assert (t.clip_count, t.zero_count, t.nan_blocks) == INCIDENT_COUNTS[(variant, rule)] + (0,)
    small_amax = {"original": 1.0, "spike": 500.0, "zero_row": 0.0}[variant]
    assert t.amax.ravel().tolist() == [small_amax, 500.0]
    assert np.array_equal(t.scales, O.quantize(x, "e4m3", "row", rule).scales)
    if variant == "original":
        # the pattern's binades, four repeats each (0.03 and 2^-6 share one, as
        # do 0.117 and 2^-4)
        want = {-10: 4, -6: 8, -4: 8, -2: 4, -1: 4, 0: 4}
        want.update({b: 4 for b in range(1, 9)})
        assert t.binades == want


def test_incident_trace_counts_nan_blocks_apart():
    x = np.full((2, 64), 1000.0)
    x[0, 5] = np.nan
    x[1, 40] = np.inf
    t = O.incident_trace(x, "e4m3", "row", "floor")
    # every finite 1000 outside the two NaN/Inf blocks is clipped (S = 2 under
    # the floor rule: 1000 / 2 = 500 > 448); the NaN and Inf blocks count apart
    assert t.nan_blocks == 2 and t.clip_count == 64 and t.zero_count == 0


@pytest.mark.parametrize("rule", ["ceil", "floor"])
def test_troubleshooting_selector_column(golden_dir, rule):
    """The selector column quantizes exactly (amax 1: S = 2^-8 under both
    rules, 1/S = 256 on the grid) and returns column 3 of X-hat: the page
    prints [0.5, 512] for the ceil rule; the floor rule saturates to 448."""
    g = load(golden_dir, "two_row_fixture.json")
    x, _ = two_row_fixture(g)
    qs = O.quantize(selector_w(), "e4m3", "col", rule=rule)
    assert O.decode_e8m0(int(qs.scales[0, 0])) == 2.0 ** -8
    assert O.dequantize(qs).ravel().tolist() == selector_w().ravel().tolist()
    ys, _ = O.gemm(O.quantize(x, "e4m3", "row", rule=rule), qs)
    if rule == "ceil":
        assert ys.ravel().tolist() == g["ceil_rule"]["selector_mx"]
    else:
        assert ys.ravel().tolist() == [0.5, 448.0]


# ---------------------------------------------------------------- GEMM

def int_operands(rng, rows, k, fmt, lim):
    """Codes of small integers (exact in the format) with scale 2^0."""
    vals = rng.integers(-lim, lim + 1, size=(rows, k)).astype(np.float64)
    codes = O.encode_sat_rne(fmt, vals)
    return vals, O.MxBlocks(codes, np.full((rows, k // 32), 127, np.uint8), O.FORMATS[fmt])


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e4m3", "e5m2")])
def test_gemm_integer_closed_form(fa, fb):
    """All scales 1 and integer codes: Y is the integer matmul (exact)."""
    rng = np.random.default_rng(7)
    av, a = int_operands(rng, 5, 96, fa, 8)
    bv, b = int_operands(rng, 3, 96, fb, 8)
    y, t = O.gemm(a, b)
    want = av.astype(np.int64) @ bv.astype(np.int64).T
    assert np.array_equal(y, want.astype(np.float64))
    assert np.array_equal(t, (np.abs(av).astype(np.int64) @ np.abs(bv).astype(np.int64).T))


def random_mx(rng, rows, k, fmt, scale_lo=110, scale_hi=140):
    t = O.decode_table(fmt)
    finite = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    codes = rng.choice(finite, size=(rows, k))
    scales = rng.integers(scale_lo, scale_hi, size=(rows, -(-k // 32))).astype(np.uint8)
    return O.MxBlocks(codes, scales, O.FORMATS[fmt])


def test_gemm_matches_exact_rational_sum():
    """Random codes and non-uniform scales: float64 oracle vs exact Fractions."""
    rng = np.random.default_rng(8)
    a = random_mx(rng, 3, 96, "e4m3")
    b = random_mx(rng, 2, 96, "e5m2")
    y, t = O.gemm(a, b)
    exact = O.exact_gemm_fraction(a, b)
    for i in range(3):
        for j in range(2):
            assert abs(Fraction(y[i, j]) - exact[i][j]) <= Fraction(t[i, j]) * Fraction(1, 2 ** 45)
    # T is the sum of |products| (brute force)
    ta, tb = O.decode_table("e4m3"), O.decode_table("e5m2")
    sa, sb = O.e8m0_values(a.scales), O.e8m0_values(b.scales)
    for i in range(3):
        for j in range(2):
            want = sum(abs(ta[a.codes[i, k]] * sa[i, k // 32] * tb[b.codes[j, k]] * sb[j, k // 32])
                       for k in range(96))
            assert abs(t[i, j] - want) <= 1e-12 * want


def test_gemm_keeps_block_scales_inside_the_sum(golden_dir):
    """Two K-blocks with partial sums 2 and 3 and scale products 4 and 8: the
    definition gives 2*4 + 3*8, not 4*(2+3) (the page's 34-vs-25 point)."""
    g = load(golden_dir, "block_sum.json")
    assert sum(p * s for p, s in zip(g["partials"], g["scale_products"])) == g["block_scaled_sum"]
    v = g["e8m0_variant"]
    a_codes = np.zeros((1, 64), np.uint8)
    b_codes = np.zeros((1, 64), np.uint8)
    one = O.encode_sat_rne("e4m3", np.array([1.0]))[0]
    a_codes[0, 0:2] = one          # block 0: partial 1 + 1 = 2
    a_codes[0, 32:35] = one        # block 1: partial 3
    b_codes[0, :] = one
    sa = np.array([[127 + 2, 127 + 3]], np.uint8)      # 4, 8
    sb = np.array([[127, 127]], np.uint8)
    y, _ = O.gemm(O.MxBlocks(a_codes, sa, O.E4M3), O.MxBlocks(b_codes, sb, O.E4M3))
    assert y[0, 0] == v["block_scaled_sum"] != v["pulled_out_sum"]


def test_gemm_block_form_equals_dequantized_matmul():
    rng = np.random.default_rng(9)
    a = random_mx(rng, 17, 160, "e4m3")
    b = random_mx(rng, 9, 160, "e4m3")
    y, t = O.gemm(a, b)
    ref = O.dequantize(a) @ O.dequantize(b).T
    assert np.all(np.abs(y - ref) <= 1e-13 * t)


def test_gemm_operand_orientation():
    """A [M,K] and B [N,K]: a transposed or swapped operand fails here."""
    rng = np.random.default_rng(10)
    av, a = int_operands(rng, 4, 64, "e4m3", 5)
    bv, b = int_operands(rng, 7, 64, "e4m3", 5)
    y, _ = O.gemm(a, b)
    assert y.shape == (4, 7)
    assert y[2, 5] == float(np.dot(av[2], bv[5]))


def test_grouped_gemm_is_per_group_dense():
    rng = np.random.default_rng(11)
    offsets = np.array([0, 0, 5, 37, 37, 40])
    a = random_mx(rng, 40, 64, "e4m3")
    bs = [random_mx(rng, 6, 64, "e4m3") for _ in range(5)]
    y, _ = O.grouped_gemm(a, offsets, bs)
    for g in range(5):
        lo, hi = offsets[g], offsets[g + 1]
        for i in range(lo, hi):
            row = O.MxBlocks(a.codes[i:i + 1], a.scales[i:i + 1], a.fmt)
            assert np.array_equal(y[i], O.gemm(row, bs[g])[0][0])


# ---------------------------------------------------------------- grouped backward

MOE_TINY_OFFSETS = np.array([0, 0, 1, 32, 65, 65, 165, 200])   # sizes 0,1,31,33,0,100,35


@pytest.mark.parametrize("fa,fb", [("e5m2", "e4m3"), ("e4m3", "e4m3")])
def test_grouped_wgrad_of_lossless_integers_is_the_integer_matmul(fa, fb):
    """Integers in [-8, 8] are exact in bf16 and MX-quantize without loss in
    both formats (at most 3 significant bits; the largest scaled value is
    7 * 2^6 = 448 for E4M3 and 7 * 2^13 = 57344 for E5M2, each format's
    maximum), so each expert's weight gradient must equal the int64 product
    dY_g^T X_g over that expert's rows alone (closed form)."""
    rng = np.random.default_rng(5)
    total = int(MOE_TINY_OFFSETS[-1])
    dy = rng.integers(-8, 9, size=(total, 40)).astype(np.float64)
    x = rng.integers(-8, 9, size=(total, 72)).astype(np.float64)
    a = O.quantize_grouped_cols(dy, MOE_TINY_OFFSETS, fa)
    b = O.quantize_grouped_cols(x, MOE_TINY_OFFSETS, fb)
    y, t = O.grouped_wgrad(a, b)
    assert y.shape == (len(MOE_TINY_OFFSETS) - 1, 40, 72)
    for g in range(len(MOE_TINY_OFFSETS) - 1):
        lo, hi = MOE_TINY_OFFSETS[g], MOE_TINY_OFFSETS[g + 1]
        ref = dy[lo:hi].astype(np.int64).T @ x[lo:hi].astype(np.int64)
        assert np.array_equal(y[g], ref.astype(np.float64)), g
        assert np.array_equal(t[g], (np.abs(dy[lo:hi]).T @ np.abs(x[lo:hi])))


def test_grouped_col_blocks_start_at_each_group():
    """A block spanning two groups would give the small values of group 1
    the scale of group 0's 2^10 entries and flush them to zero; blocks that
    start at each group's first row keep them exactly."""
    offsets = np.array([0, 5, 45])
    x = np.zeros((45, 32))
    x[:5] = 2.0 ** 10
    rng = np.random.default_rng(2)
    x[5:] = rng.integers(1, 8, size=(40, 32)) * 2.0 ** -10
    q = O.quantize_grouped_cols(x, offsets, "e4m3")
    deq = O.dequantize(q[1])            # [32 columns, 64 padded tokens]
    assert np.array_equal(deq[:, :40], x[5:].T)
    assert np.all(deq[:, 40:] == 0)


def test_grouped_col_partial_block_is_zero_padded():
    """A group of 33 rows has two blocks; the second holds one real row and
    31 zeros, so its scale is the floor rule applied to that row alone
    (frexp closed form) and its padding codes are +0."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((33, 64)) * 3
    q = O.quantize_grouped_cols(x, [0, 33], "e4m3")[0]
    assert q.codes.shape == (64, 64)
    assert np.all(q.codes[:, 33:] == 0)
    for c in range(64):
        _, ex = math.frexp(abs(x[32, c]))      # |x| = f * 2^ex, f in [0.5, 1)
        assert q.scales[c, 1] == (ex - 1) - 8 + 127


# ------------------------------------------- partial final blocks (K % 32 != 0)


def test_partial_final_block_worked_example():
    """K = 48: a whole block of ones, then a 16-element block whose amax is 3.
    By hand (E4M3, floor rule): block 0 has e = 0 - 8, scale byte 119, and
    1 * 2^8 = 256 = 1.0 * 2^8 is code (8 + 7) << 3 = 0x78; block 1 has
    e = floor(log2 3) - 8 = -7, scale byte 120, 3 * 2^7 = 384 = 1.5 * 2^8 is
    code 0x78 | 4 = 0x7C, -0.75 * 2^7 = -96 = -1.5 * 2^6 is code
    0x80 | (6 + 7) << 3 | 4 = 0xEC, and 0.5 * 2^7 = 64 = 2^6 is 0x68.  The
    same values down a column give the same codes and scales."""
    x = np.zeros((1, 48))
    x[0, :32] = 1.0
    x[0, 32:36] = [3.0, -0.75, 0.0, 0.5]
    q = O.quantize(x, "e4m3", "row")
    assert q.codes.shape == (1, 48) and q.scales.shape == (1, 2)
    assert list(q.scales[0]) == [119, 120]
    assert np.all(q.codes[0, :32] == 0x78)
    assert list(q.codes[0, 32:36]) == [0x7C, 0xEC, 0x00, 0x68]
    assert np.all(q.codes[0, 36:] == 0)
    c = O.quantize(x.T.copy(), "e4m3", "col")
    assert np.array_equal(c.codes, q.codes) and np.array_equal(c.scales, q.scales)


@pytest.mark.parametrize("k", [16, 48, 80, 112])
def test_partial_block_takes_the_floor_rule_of_its_own_values(k):
    """The final block's scale is the floor rule applied to its K % 32 real
    values (frexp closed form), and its codes are torch's saturating E4M3
    cast of those values over the scale."""
    rng = np.random.default_rng(k)
    x = rng.standard_normal((6, k)) * np.exp2(rng.integers(-10, 10, size=(6, 1)))
    x = torch.tensor(x).to(torch.bfloat16).double().numpy()
    q = O.quantize(x, "e4m3", "row")
    last = k // 32
    assert q.scales.shape == (6, last + 1)
    for r in range(6):
        _, ex = math.frexp(float(np.max(np.abs(x[r, 32 * last:]))))
        e = (ex - 1) - 8
        assert q.scales[r, last] == e + 127
        scaled = torch.tensor(x[r, 32 * last:] * 2.0 ** -e).clamp(-448, 448)
        want = scaled.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q.codes[r, 32 * last:], want)


@pytest.mark.parametrize("k", [16, 48, 208])
def test_ragged_k_gemm_of_lossless_integers_is_the_integer_matmul(k):
    """Integers in [-4, 4], each block holding a 4 or a -4: every value
    quantizes exactly (v * 2^6 is an E4M3 value), so the GEMM over K
    elements, partial final block included, is the integer matmul."""
    rng = np.random.default_rng(k + 1)
    av = rng.integers(-4, 5, size=(5, k))
    bv = rng.integers(-4, 5, size=(3, k))
    for m in (av, bv):
        m[:, ::32] = 4
    a = O.quantize(av.astype(np.float64), "e4m3", "row")
    b = O.quantize(bv.astype(np.float64), "e4m3", "row")
    y, t = O.gemm(a, b)
    assert np.array_equal(y, (av @ bv.T).astype(np.float64))
    assert np.array_equal(t, (np.abs(av) @ np.abs(bv).T).astype(np.float64))


def test_ragged_k_gemm_matches_exact_rational_sum():
    """K = 80 (two whole blocks and a 16-element one), random codes and
    scales: float64 oracle vs exact Fractions, and T by brute force."""
    rng = np.random.default_rng(18)
    a = random_mx(rng, 3, 80, "e4m3")
    b = random_mx(rng, 2, 80, "e5m2")
    assert a.scales.shape == (3, 3)
    y, t = O.gemm(a, b)
    exact = O.exact_gemm_fraction(a, b)
    ta, tb = O.decode_table("e4m3"), O.decode_table("e5m2")
    sa, sb = O.e8m0_values(a.scales), O.e8m0_values(b.scales)
    for i in range(3):
        for j in range(2):
            assert abs(Fraction(y[i, j]) - exact[i][j]) <= Fraction(t[i, j]) * Fraction(1, 2 ** 45)
            want = sum(abs(ta[a.codes[i, kk]] * sa[i, kk // 32] * tb[b.codes[j, kk]] * sb[j, kk // 32])
                       for kk in range(80))
            assert abs(t[i, j] - want) <= 1e-12 * want


def test_ragged_k_equals_the_zero_extended_k():
    """The page's zero-padded final block: quantizing and multiplying K = 48
    columns gives the codes, scales and product of the same data extended
    with 16 zero columns (the padding's codes are +0)."""
    rng = np.random.default_rng(19)
    x = rng.standard_normal((4, 48))
    w = rng.standard_normal((3, 48)) * 0.1
    xp = np.concatenate([x, np.zeros((4, 16))], axis=1)
    wp = np.concatenate([w, np.zeros((3, 16))], axis=1)
    for fmt in ("e4m3", "e2m1"):
        a, ap = O.quantize(x, fmt, "row"), O.quantize(xp, fmt, "row")
        b, bp = O.quantize(w, fmt, "row"), O.quantize(wp, fmt, "row")
        assert np.array_equal(a.scales, ap.scales) and np.array_equal(a.codes, ap.codes[:, :48])
        assert np.all(ap.codes[:, 48:] == 0)
        assert np.array_equal(O.gemm(a, b)[0], O.gemm(ap, bp)[0])


def test_stacked_weights_colwise_equal_per_expert_operands():
    """dgrad operand of a mixture of experts: with N % 32 == 0, columnwise
    blocks of the stacked [E*N, K] weights never span two experts, so one
    columnwise quantization of the stack is the per-expert quantizations
    side by side along K (columns [g*N, (g+1)*N))."""
    rng = np.random.default_rng(4)
    e, n, k = 3, 64, 96
    w = rng.standard_normal((e, n, k)) * 0.02
    whole = O.quantize(w.reshape(e * n, k), "e4m3", "col")
    for g in range(e):
        part = O.quantize(w[g], "e4m3", "col")
        assert np.array_equal(whole.codes[:, g * n:(g + 1) * n], part.codes)
        assert np.array_equal(whole.scales[:, g * n // 32:(g + 1) * n // 32], part.scales)


def test_pack_grouped_cols_layout():
    """Each group starts at a 128-column boundary, the segments do not
    overlap, and unpacking returns every group's codes and scales."""
    rng = np.random.default_rng(6)
    total = int(MOE_TINY_OFFSETS[-1])
    x = rng.standard_normal((total, 24))
    qs = O.quantize_grouped_cols(x, MOE_TINY_OFFSETS, "e5m2")
    starts = O.grouped_scale_rows(MOE_TINY_OFFSETS)
    assert list(starts) == [0, 0, 128, 256, 384, 384, 512, 640]
    codes, scales = O.pack_grouped_cols(qs, MOE_TINY_OFFSETS, 768)
    for g, q in enumerate(qs):
        s0, kp = int(starts[g]), q.codes.shape[1]
        assert np.array_equal(codes[:, s0:s0 + kp], q.codes)
        assert np.array_equal(scales[:, s0 // 32:(s0 + kp) // 32], q.scales)
        assert np.all(codes[:, s0 + kp:int(starts[g + 1])] == 0)
    with pytest.raises(ValueError):
        O.pack_grouped_cols(qs, MOE_TINY_OFFSETS, 512)


# ---------------------------------------------------------------- MXFP6 / MXFP4 element formats

NARROW = ["e2m3", "e3m2", "e2m1"]


@pytest.mark.parametrize("fmt", NARROW)
def test_narrow_formats_from_page(golden_dir, fmt):
    """Maxima printed on the page pin each format's (ebits, mbits, bias);
    the grid has no Inf or NaN, 2^(bits-1) - 1 positive values, and within
    every binade 2^mbits equal steps that double at each binade boundary."""
    g = load(golden_dir, "mx_narrow_formats.json")
    f = O.fmt_of(fmt)
    t = O.decode_table(f)
    assert len(t) == 1 << f.bits and np.isfinite(t).all()
    assert t.max() == g[fmt]["max"] == f.max_finite and t.min() == -g[fmt]["max"]
    pos = np.unique(t[t > 0])
    assert len(pos) == (1 << (f.bits - 1)) - 1
    # below the smallest normal: the subnormals k * step, k = 1 .. 2^mbits - 1
    sub = pos[pos < f.min_normal]
    assert np.array_equal(sub, f.subnormal_step * np.arange(1, 1 << f.mbits))
    # every normal binade [2^e, 2^(e+1)) up to the top one: 2^mbits values
    # spaced 2^(e - mbits), the spacing doubling from binade to binade
    e = 1 - f.bias
    while 2.0 ** e <= f.max_finite:
        inside = pos[(pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1))]
        assert np.array_equal(inside, 2.0 ** e + 2.0 ** (e - f.mbits) * np.arange(1 << f.mbits))
        e += 1
    assert e - 1 == f.emax_elem
    assert O.BLOCK == g["block"]


def test_e2m1_values():
    """E2M1 (sign, 2 exponent bits with bias 1, 1 mantissa bit): the eight
    magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, and their negatives."""
    t = O.decode_table("e2m1")
    assert list(t[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(t[8:]) == [-v for v in t[:8]]
    assert np.signbit(t[8]) and not np.signbit(t[0])


def brute_force_encode(fmt, v):
    """Nearest finite code by exhaustive search; ties to the even code (the
    code whose last mantissa bit is 0); a negative value that rounds to zero
    keeps its sign."""
    f = O.fmt_of(fmt)
    t = O.decode_table(f)
    codes = np.arange(len(t))
    out = np.empty(len(v), dtype=np.uint8)
    for i, x in enumerate(v):
        d = np.abs(t - x)
        best = codes[d == d.min()]
        best = [c for c in best if (t[c] != 0 or np.signbit(t[c]) == np.signbit(x))] or list(best)
        if len(best) > 1:
            even = [c for c in best if c % 2 == 0]
            best = even or best
        out[i] = best[0]
    return out


@pytest.mark.parametrize("fmt", NARROW)
def test_narrow_encode_matches_brute_force(fmt):
    f = O.fmt_of(fmt)
    rng = np.random.default_rng(hash(fmt) % 1000)
    t = O.decode_table(f)
    mids = (np.sort(np.unique(t))[1:] + np.sort(np.unique(t))[:-1]) / 2   # every tie point
    v = np.concatenate([rng.standard_normal(3000) * f.max_finite / 3,
                        rng.standard_normal(500) * f.subnormal_step * 4,
                        mids, t, [f.max_finite * 1.01, -f.max_finite * 9, 1e-30, -1e-30]])
    got = O.encode_sat_rne(f, v)
    want = brute_force_encode(f, v)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", NARROW)
def test_narrow_block_scale_rules(fmt):
    """Floor rule: the scaled amax lands in the top binade [2^emax,
    2^(emax+1)); ceil rule: brute-force smallest e with amax <= max * 2^e."""
    f = O.fmt_of(fmt)
    rng = np.random.default_rng(7)
    amax = np.exp(rng.uniform(-30, 30, 2000))
    e = O.scale_exponent_floor(f, amax)
    scaled = amax / 2.0 ** e
    assert np.all((scaled >= 2.0 ** f.emax_elem) & (scaled < 2.0 ** (f.emax_elem + 1)))
    c = O.scale_exponent_ceil(f, amax)
    for a, ec in zip(amax[:300], c[:300]):
        want = min(k for k in range(-140, 140) if a <= f.max_finite * 2.0 ** k)
        assert ec == want


def test_narrow_quantize_nan_block_writes_zero_codes():
    x = np.ones((1, 64))
    x[0, 5] = np.nan
    q = O.quantize(x, "e2m1", "row")
    assert q.scales[0, 0] == 0xFF and np.all(q.codes[0, :32] == 0)
    assert q.scales[0, 1] == 127 - 2 and np.all(O.decode_table("e2m1")[q.codes[0, 32:]] == 4.0)


@pytest.mark.parametrize("fmt", NARROW + ["e4m3"])
def test_container_round_trip(fmt):
    """Packing keeps 16 codes per 16 bytes (FP8: identity) and unpacks to
    the same codes; the padding bytes are zero."""
    f = O.fmt_of(fmt)
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 1 << f.bits, size=(5, 64)).astype(np.uint8)
    buf = O.pack_container(codes, f)
    assert buf.shape == codes.shape
    assert np.array_equal(O.unpack_container(buf, f), codes)
    if f.bits < 8:
        used = 2 * f.bits
        assert np.all(buf.reshape(5, 4, 16)[:, :, used:] == 0)


# ---------------------------------------------------------------- swizzle

@pytest.mark.parametrize("fmt", ["e2m3", "e3m2", "e2m1"])
def test_dense_packing(fmt):
    """Packed storage of the narrow codes: every code comes back out
    (round trip over random codes of every value), the byte count is the
    page's payload (K * w / 8 per row), the E2M1 nibble order is element 2i
    in the low nibble of byte i, and each 16-element run's packed bytes are
    exactly the container's first 8 (E2M1) or 12 (E2M3, E3M2) bytes."""
    f = O.fmt_of(fmt)
    rng = np.random.default_rng(17)
    codes = rng.integers(0, 1 << f.bits, size=(5, 128), dtype=np.uint8)
    packed = O.pack_dense(codes, fmt)
    assert packed.shape == (5, 128 * f.bits // 8)
    assert np.array_equal(O.unpack_dense(packed, fmt), codes)
    runs = O.pack_container(codes, fmt).reshape(5, 8, 16)[:, :, :2 * f.bits]
    assert np.array_equal(runs.reshape(5, -1), packed)
    if f.bits == 4:
        assert np.array_equal(packed & 0xF, codes[:, 0::2])
        assert np.array_equal(packed >> 4, codes[:, 1::2])
    else:  # four 6-bit codes a, b, c, d in three bytes, little-endian
        a, b, c, d = (codes[:, i::4].astype(np.uint32) for i in range(4))
        assert np.array_equal(packed[:, 0::3], (a | (b & 3) << 6).astype(np.uint8))
        assert np.array_equal(packed[:, 1::3], (b >> 2 | (c & 15) << 4).astype(np.uint8))
        assert np.array_equal(packed[:, 2::3], (c >> 4 | d << 2).astype(np.uint8))
    # every code value in every position of a 16-element run
    allc = np.array([[(v + i) % (1 << f.bits) for i in range(16)] for v in range(1 << f.bits)],
                    dtype=np.uint8)
    assert np.array_equal(O.unpack_dense(O.pack_dense(allc, fmt), fmt), allc)


@pytest.mark.parametrize("rows,kb", [(1, 1), (128, 4), (130, 5), (300, 17), (256, 224)])
def test_swizzle_is_a_bijection_and_round_trips(rows, kb):
    size = O.scale_bytes(rows, kb)
    r, c = np.meshgrid(np.arange(-(-rows // 128) * 128), np.arange(-(-kb // 4) * 4), indexing="ij")
    off = O.swizzle_offset(r, c, kb).ravel()
    assert np.array_equal(np.sort(off), np.arange(size))
    rng = np.random.default_rng(rows * 1000 + kb)
    s = rng.integers(0, 255, size=(rows, kb)).astype(np.uint8)
    buf = O.swizzle_scales(s)
    assert buf.size == size
    assert np.array_equal(O.unswizzle_scales(buf, rows, kb), s)
    mask = np.ones(size, bool)
    mask[O.swizzle_offset(*np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij"), kb).ravel()] = False
    assert np.all(buf[mask] == 0)


def test_swizzle_tile_structure():
    """Each 128x4 tile is one contiguous 512-byte unit; 32-row groups of a
    tile interleave at 4-byte slots of 16-byte lines."""
    kb = 8
    assert O.swizzle_offset(0, 0, kb) == 0
    assert O.swizzle_offset(0, 4, kb) == 512
    assert O.swizzle_offset(128, 0, kb) == 1024
    assert O.swizzle_offset(1, 0, kb) == 16
    assert O.swizzle_offset(32, 0, kb) == 4
    assert O.swizzle_offset(0, 3, kb) == 3


def test_grouped_swizzle_places_each_group_at_a_tile_boundary():
    rng = np.random.default_rng(12)
    offsets = np.array([0, 3, 3, 200, 201, 460])
    s = rng.integers(0, 255, size=(460, 8)).astype(np.uint8)
    buf = O.swizzle_scales_grouped(s, offsets)
    starts = O.grouped_scale_rows(offsets)
    assert starts.tolist() == [0, 128, 128, 384, 512, 896]
    assert buf.size >= O.scale_bytes(starts[-1], 8)
    for g in range(5):
        lo, hi = offsets[g], offsets[g + 1]
        if lo == hi:
            continue
        base = starts[g] // 128 * 2 * 512
        part = buf[base:base + O.scale_bytes(hi - lo, 8)]
        assert np.array_equal(O.unswizzle_scales(part, hi - lo, 8), s[lo:hi])


# ---------------------------------------------------------------- fused epilogue

def test_silu_matches_torch_and_identities():
    """SiLU against torch's float64 silu (library routine), plus closed forms:
    silu(0) = 0, silu(z) - silu(-z) = z, silu(z) -> z for large z, -> -0
    for very negative z."""
    z = np.concatenate([np.linspace(-30, 30, 2001), [-1e4, 1e4, 0.0]])
    mine = O.silu(z)
    ref = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    assert np.allclose(mine, ref, rtol=1e-15, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(O.silu(z) - O.silu(-z), z, rtol=1e-14, atol=1e-14)
    assert O.silu(np.array([1e4]))[0] == 1e4
    assert O.silu(np.array([-1e4]))[0] == 0.0


def test_bias_is_an_extra_k_block_of_ones():
    """Y + bias equals the block-scaled GEMM with one more K-block in which A
    holds 1.0 in its first column and B holds the bias there (bias values
    chosen exactly representable)."""
    rng = np.random.default_rng(13)
    m, n, k = 6, 5, 64
    av = rng.integers(-5, 6, size=(m, k)).astype(np.float64)
    bv = rng.integers(-5, 6, size=(n, k)).astype(np.float64)
    bias = rng.integers(-7, 8, size=n).astype(np.float64) * 0.25
    a = O.MxBlocks(O.encode_sat_rne("e4m3", av), np.full((m, 2), 127, np.uint8), O.E4M3)
    b = O.MxBlocks(O.encode_sat_rne("e4m3", bv), np.full((n, 2), 127, np.uint8), O.E4M3)
    out, z, _ = O.gemm_bias_act(a, b, bias, "none")
    a2 = np.zeros((m, k + 32))
    a2[:, :k] = av
    a2[:, k] = 1.0
    b2 = np.zeros((n, k + 32))
    b2[:, :k] = bv
    b2[:, k] = bias
    qa = O.MxBlocks(O.encode_sat_rne("e4m3", a2), np.full((m, 3), 127, np.uint8), O.E4M3)
    qb = O.MxBlocks(O.encode_sat_rne("e4m3", b2), np.full((n, 3), 127, np.uint8), O.E4M3)
    y2, _ = O.gemm(qa, qb)
    assert np.array_equal(out, y2) and np.array_equal(z, y2)
    act, _, _ = O.gemm_bias_act(a, b, bias, "silu")
    assert np.array_equal(act, O.silu(y2))


# ---------------------------------------------------------------- stochastic rounding

def test_stochastic_rounding_probability_from_page(golden_dir):
    """Page's Fraction example: neighbours 1 and 9/8, x = 1.01, probability of
    rounding up 2/25.  With 16-bit draws, exactly floor(2/25 * 2^16) of the
    2^16 values round up (x = 1.01 is not dyadic, so the count is checked
    against the exact fraction of its float64 value)."""
    x = np.full(1 << 16, 1.01)
    r = np.arange(1 << 16)
    vals = O.decode_table("e4m3")[O.encode_sat_sr("e4m3", x, r)]
    assert set(vals.tolist()) == {1.0, 1.125}
    ups = int((vals == 1.125).sum())
    frac = (Fraction(1.01) - 1) / Fraction(1, 8)
    assert abs(frac - Fraction(2, 25)) < Fraction(1, 10 ** 15)
    assert ups == int(frac * (1 << 16))
    assert abs(ups / (1 << 16) - 2 / 25) < 2 ** -16


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m3", "e3m2", "e2m1"])
def test_stochastic_rounding_is_unbiased_for_dyadic_inputs(fmt):
    """E[SR(x)] = x exactly over all 2^16 draws when the fraction of a grid
    step has at most 16 bits (closed form), and grid values never move."""
    rng = np.random.default_rng(17)
    t = O.decode_table(fmt)
    grid = np.sort(t[np.isfinite(t) & (t > 0) & (t < O.FORMATS[fmt].max_finite)])
    r = np.arange(1 << 16)
    for _ in range(40):
        i = rng.integers(0, grid.size - 1)
        lo, hi = grid[i], grid[i + 1]
        x = lo + (hi - lo) * rng.integers(0, 1 << 16) / (1 << 16)
        vals = t[O.encode_sat_sr(fmt, np.full(1 << 16, x), r)]
        assert set(np.unique(vals)) <= {lo, hi}
        assert np.mean(vals) == x
        neg = t[O.encode_sat_sr(fmt, np.full(1 << 16, -x), r)]
        assert np.array_equal(neg, -vals)
    for g in grid[::7]:
        assert np.all(t[O.encode_sat_sr(fmt, np.full(64, g), np.arange(64) * 1000)] == g)


def test_stochastic_rounding_saturates_and_keeps_signed_zero():
    t = O.decode_table("e4m3")
    r = np.array([0, 65535])
    assert np.all(t[O.encode_sat_sr("e4m3", np.array([470.0, 470.0]), r)] == 448.0)
    z = O.encode_sat_sr("e4m3", np.array([-2.0 ** -30, -2.0 ** -30]), r)
    assert np.all(z == 0x80)
    assert O.encode_sat_sr("e4m3", np.array([np.nan]), np.array([0]))[0] == O.NAN_CODE


def test_stochastic_rounding_of_mxfp4_codes():
    """E2M1 (grid 0, 0.5, 1, 1.5, 2, 3, 4, 6): 5.5 lies a quarter step below
    6 and goes up for 3/4 of the draws; 0.25 (half the subnormal step 0.5)
    for half of them; 7 lies past the maximum and saturates to 6 for every
    draw (its neighbours 6 and 8, the grid extended one step); -0.1 rounds
    to -0 or -0.5 and keeps its sign."""
    t = O.decode_table("e2m1")
    r = np.arange(1 << 16)
    up = t[O.encode_sat_sr("e2m1", np.full(1 << 16, 5.5), r)]
    assert set(up.tolist()) == {4.0, 6.0} and int((up == 6.0).sum()) == 3 * (1 << 14)
    half = t[O.encode_sat_sr("e2m1", np.full(1 << 16, 0.25), r)]
    assert set(half.tolist()) == {0.0, 0.5} and int((half == 0.5).sum()) == 1 << 15
    assert np.all(t[O.encode_sat_sr("e2m1", np.full(1 << 16, 7.0), r)] == 6.0)
    neg = O.encode_sat_sr("e2m1", np.full(1 << 16, -0.1), r)
    assert set(t[neg].tolist()) == {-0.0, -0.5} and np.all(neg & 0x8)


def test_stochastic_quantize_uses_the_same_scales_as_rne():
    """Scales depend only on amax; codes differ from RNE by at most one grid
    step and equal RNE where the value is on the grid."""
    rng = np.random.default_rng(19)
    x = rng.standard_normal((32, 128)) * 3
    x = O.bf16_bits_to_float64((x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    rand = rng.integers(0, 1 << 16, size=x.shape)
    for axis in ("row", "col"):
        q = O.quantize(x, "e4m3", axis)
        s = O.quantize(x, "e4m3", axis, rand=rand)
        assert np.array_equal(q.scales, s.scales)
        dq, ds = O.dequantize(q), O.dequantize(s)
        assert np.all(np.abs(dq - ds) <= np.abs(dq) / 8 + 2.0 ** -9 * O.e8m0_values(q.scales).repeat(32, axis=1))


@pytest.mark.parametrize("rule", ["floor", "ceil"])
def test_block_amax_is_a_magnitude(rule):
    """A block whose largest magnitude is negative: the scale follows |x|,
    not the signed maximum (floor rule: floor(log2 500) - 8 = 0, byte 127;
    ceil rule: ceil(log2(500 / 448)) = 1, byte 128), and -500 comes back as
    -448 (floor: saturated at S = 1) or -512 (ceil: -250 rounds to the code
    -256 at S = 2)."""
    x = np.array([[-500.0, 1.0, 2.0, 3.0] + [0.5] * 28,
                  [-1.0] * 32], dtype=np.float64)
    q = O.quantize(x, "e4m3", "row", rule)
    assert q.scales[0, 0] == (127 if rule == "floor" else 128)
    # an all-negative block: amax 1 -> scale 2^-8 under both rules
    assert q.scales[1, 0] == 119
    xh = O.dequantize(q)
    assert xh[0, 0] == (-448.0 if rule == "floor" else -512.0)
    assert xh[1].tolist() == [-1.0] * 32
