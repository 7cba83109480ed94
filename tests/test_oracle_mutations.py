"""Planted mistakes: each test plants one plausible bug in the oracle (on the
CPU, by replacing one oracle function for the duration of the test) and
checks that the pins of tests/test_oracle.py catch it -- a dropped term, a
wrong sign, index or bound, a transposed operand, a wrong rounding or scale
rule.  A mutant counts as caught when at least one of the named pins fails.
Test infrastructure; imports the oracle."""
import math
import os

import numpy as np

import test_oracle as T
from mxcheck import ROOT
from oracle import mx_oracle as O

GOLDEN = os.path.join(ROOT, "tests", "golden")


def caught(*pins) -> bool:
    """True if at least one pin (a zero-argument callable) fails."""
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def test_pins_pass_on_the_unmodified_oracle():
    assert not caught(lambda: T.test_decode_all_codes_match_torch("e4m3"),
                      lambda: T.test_midpoints_tie_to_even_code("e4m3"),
                      lambda: T.test_gemm_keeps_block_scales_inside_the_sum(GOLDEN),
                      lambda: T.test_swizzle_tile_structure(),
                      lambda: T.test_stochastic_rounding_probability_from_page(GOLDEN))


def test_wrong_exponent_bias_in_decode(monkeypatch):
    good = O.decode_code

    def bad(fmt, code):
        v = good(fmt, code)
        return v * 2.0 if math.isfinite(v) else v      # bias one too small
    monkeypatch.setattr(O, "decode_code", bad)
    assert caught(lambda: T.test_decode_all_codes_match_torch("e4m3"),
                  lambda: T.test_format_facts_from_page(GOLDEN))


def test_ties_away_from_zero_instead_of_to_even(monkeypatch):
    def bad(fmt, v):
        f = O.fmt_of(fmt)
        v = np.asarray(v, dtype=np.float64)
        a = np.abs(v)
        _, ex = np.frexp(a)
        qe = np.where(a < f.min_normal, 1 - f.bias - f.mbits, ex.astype(np.int64) - 1 - f.mbits)
        return np.copysign(np.ldexp(np.floor(np.ldexp(a, -qe) + 0.5), qe), v)
    monkeypatch.setattr(O, "round_to_grid_rne", bad)
    assert caught(lambda: T.test_midpoints_tie_to_even_code("e4m3"),
                  lambda: T.test_cast_audit_from_page(GOLDEN))


def test_missing_saturation(monkeypatch):
    def bad(fmt, v):
        f = O.fmt_of(fmt)
        r = O.round_to_grid_rne(f, np.where(np.isfinite(v), v, 0.0))
        r = np.where(np.abs(r) > f.max_finite, np.copysign(2.0 ** -9, r), r)  # no clamp to max
        return O.encode_grid_value(f, r)
    monkeypatch.setattr(O, "encode_sat_rne", bad)
    assert caught(lambda: T.test_saturation_and_rne_from_page(GOLDEN),
                  lambda: T.test_cast_audit_from_page(GOLDEN))


def test_negative_underflow_loses_its_sign(monkeypatch):
    good = O.round_to_grid_rne
    monkeypatch.setattr(O, "round_to_grid_rne", lambda fmt, v: np.abs(good(fmt, v)) *
                        np.where(good(fmt, v) == 0, 1.0, np.sign(good(fmt, v))))
    assert caught(lambda: T.test_cast_audit_from_page(GOLDEN),
                  lambda: T.test_encode_is_monotone_and_keeps_sign("e4m3"))


def test_scale_rule_emax_off_by_one(monkeypatch):
    good = O.scale_exponent_floor
    monkeypatch.setattr(O, "scale_exponent_floor", lambda fmt, amax: np.clip(
        good(fmt, amax) + 1, -127, 127))
    assert caught(lambda: T.test_floor_rule_puts_scaled_amax_in_top_binade(),
                  lambda: T.test_two_row_experiment_floor_rule_saturates_spike(GOLDEN))


def test_ceil_rule_replaced_by_the_floor_rule(monkeypatch):
    monkeypatch.setattr(O, "scale_exponent_ceil", O.scale_exponent_floor)
    assert caught(lambda: T.test_ceil_rule_brute_force(),
                  lambda: T.test_two_row_experiment_ceil_rule_from_page(GOLDEN))


def _gemm_variant(transform):
    def bad(a, b):
        m, k = a.codes.shape
        n = b.codes.shape[0]
        nb = k // O.BLOCK
        av = O.decode_table(a.fmt)[a.codes].reshape(m, nb, O.BLOCK)
        bv = O.decode_table(b.fmt)[b.codes].reshape(n, nb, O.BLOCK)
        sa, sb = O.e8m0_values(a.scales), O.e8m0_values(b.scales)
        return transform(av, bv, sa, sb, m, n, nb)
    return bad


def test_block_scales_pulled_out_of_the_sum(monkeypatch):
    def t(av, bv, sa, sb, m, n, nb):
        # one scale product per output (the first block's) times the raw sum
        raw = sum(av[:, i, :] @ bv[:, i, :].T for i in range(nb))
        y = sa[:, 0][:, None] * sb[:, 0][None, :] * raw
        return y, np.abs(y) + 1.0
    monkeypatch.setattr(O, "gemm", _gemm_variant(t))
    assert caught(lambda: T.test_gemm_keeps_block_scales_inside_the_sum(GOLDEN),
                  lambda: T.test_gemm_matches_exact_rational_sum())


def test_last_k_block_dropped(monkeypatch):
    def t(av, bv, sa, sb, m, n, nb):
        y = np.zeros((m, n))
        for i in range(nb - 1):
            y += sa[:, i][:, None] * sb[:, i][None, :] * (av[:, i, :] @ bv[:, i, :].T)
        return y, np.abs(y) + 1.0
    monkeypatch.setattr(O, "gemm", _gemm_variant(t))
    assert caught(lambda: T.test_gemm_matches_exact_rational_sum(),
                  lambda: T.test_gemm_integer_closed_form("e4m3", "e4m3"))


def test_gemm_result_transposed(monkeypatch):
    good = O.gemm
    monkeypatch.setattr(O, "gemm", lambda a, b: tuple(z.T for z in good(a, b)))
    assert caught(lambda: T.test_gemm_operand_orientation())


def test_gemm_b_decoded_with_a_format(monkeypatch):
    good = O.gemm
    monkeypatch.setattr(O, "gemm", lambda a, b: good(a, O.MxBlocks(b.codes, b.scales, a.fmt)))
    assert caught(lambda: T.test_gemm_integer_closed_form("e4m3", "e5m2"))


def test_swizzle_row_roles_swapped(monkeypatch):
    def bad(r, c, kblocks):
        r = np.asarray(r, dtype=np.int64)
        c = np.asarray(c, dtype=np.int64)
        tiles_k = -(-kblocks // O.TILE_BLOCKS)
        tile = (r // O.TILE_ROWS) * tiles_k + c // O.TILE_BLOCKS
        inner = ((r % O.TILE_ROWS) // 32) * 128 + (r % 32) * 4 + c % O.TILE_BLOCKS
        return tile * O.TILE_BYTES + inner
    monkeypatch.setattr(O, "swizzle_offset", bad)
    assert caught(lambda: T.test_swizzle_tile_structure())


def test_stochastic_rounding_compare_off_by_one(monkeypatch):
    def bad(fmt, v, rand):
        f = O.fmt_of(fmt)
        v = np.asarray(v, dtype=np.float64)
        a = np.abs(v)
        _, ex = np.frexp(a)
        qe = np.where(a < f.min_normal, 1 - f.bias - f.mbits, ex.astype(np.int64) - 1 - f.mbits)
        units = np.ldexp(a, -qe)
        low = np.floor(units)
        frac16 = np.floor((units - low) * 2.0 ** O.SR_BITS)
        up = np.asarray(rand, dtype=np.int64) <= frac16          # <= instead of <
        return np.copysign(np.ldexp(low + up, qe), v)
    monkeypatch.setattr(O, "round_to_grid_stochastic", bad)
    assert caught(lambda: T.test_stochastic_rounding_probability_from_page(GOLDEN),
                  lambda: T.test_stochastic_rounding_is_unbiased_for_dyadic_inputs("e4m3"))


def test_grouped_column_blocks_start_at_token_zero(monkeypatch):
    def bad(x, offsets, fmt, rule="floor"):
        # blocks counted from the first token of all experts, then sliced
        x = np.asarray(x, dtype=np.float64)
        offsets = np.asarray(offsets, dtype=np.int64)
        total = x.shape[0]
        padded = np.zeros((-(-total // O.BLOCK) * O.BLOCK, x.shape[1]))
        padded[:total] = x
        whole = O.quantize(padded, fmt, "col", rule)
        out = []
        for g in range(len(offsets) - 1):
            lo, hi = int(offsets[g]), int(offsets[g + 1])
            width = -(-(hi - lo) // O.BLOCK) * O.BLOCK
            codes = np.zeros((x.shape[1], width), np.uint8)
            codes[:, :hi - lo] = whole.codes[:, lo:hi]
            scales = whole.scales[:, lo // O.BLOCK:lo // O.BLOCK + width // O.BLOCK]
            if scales.shape[1] < width // O.BLOCK:
                scales = np.pad(scales, ((0, 0), (0, width // O.BLOCK - scales.shape[1])),
                                constant_values=127)
            out.append(O.MxBlocks(codes, scales, whole.fmt))
        return out
    monkeypatch.setattr(O, "quantize_grouped_cols", bad)
    assert caught(lambda: T.test_grouped_col_blocks_start_at_each_group(),
                  lambda: T.test_grouped_wgrad_of_lossless_integers_is_the_integer_matmul(
                      "e4m3", "e4m3"))


def test_columnwise_blocks_taken_along_the_wrong_axis(monkeypatch):
    good = O.quantize_rows

    def bad(x, fmt, axis, rule="floor", rand=None):
        x = np.asarray(x, dtype=np.float64)
        if axis == "col":       # quantized along rows, then transposed
            q = good(x, fmt, rule)
            return O.MxBlocks(q.codes.T.copy(), q.scales, q.fmt)
        return good(x, fmt, rule, rand)
    monkeypatch.setattr(O, "quantize", bad)
    assert caught(lambda: T.test_column_blocks_run_along_rows())


def test_silu_with_the_wrong_sign(monkeypatch):
    def bad(z):
        z = np.asarray(z, np.float64)
        with np.errstate(over="ignore"):
            return z / (1.0 + np.exp(z))
    monkeypatch.setattr(O, "silu", bad)
    monkeypatch.setitem(O.ACTIVATIONS, "silu", O.silu)
    assert caught(lambda: T.test_silu_matches_torch_and_identities())


def test_block_amax_takes_the_signed_maximum(monkeypatch):
    """amax = max(x) instead of max(|x|): the scale of a block led by a
    negative value is far too small."""
    good = O.quantize_rows

    def bad(x, fmt, rule="floor", rand=None):
        x = np.asarray(x, dtype=np.float64)
        rows, k = x.shape
        blocks = x.reshape(rows, k // 32, 32)
        signed_max = np.max(np.where(np.isfinite(blocks), blocks, 0.0), axis=2)
        # rescale every block so that its |x| maximum equals the signed one,
        # which is what a scale taken from max(x) quantizes against
        mag = np.max(np.abs(np.where(np.isfinite(blocks), blocks, 0.0)), axis=2)
        ratio = np.where((mag > 0) & (signed_max > 0), signed_max / np.where(mag > 0, mag, 1), 1.0)
        q = good(x, fmt, rule, rand)
        f = O.fmt_of(fmt)
        e = (O.scale_exponent_floor(f, mag * ratio) if rule == "floor"
             else O.scale_exponent_ceil(f, mag * ratio))
        scaled = np.ldexp(np.where(np.isfinite(blocks), blocks, 0.0), -e[:, :, None])
        codes = O.encode_sat_rne(f, scaled).reshape(rows, k).astype(np.uint8)
        return O.MxBlocks(codes, (e + 127).astype(np.uint8), q.fmt)
    monkeypatch.setattr(O, "quantize_rows", bad)
    assert caught(lambda: T.test_block_amax_is_a_magnitude("floor"),
                  lambda: T.test_block_amax_is_a_magnitude("ceil"))


def test_partial_block_padding_placed_in_front(monkeypatch):
    """The zeros of a partial final block put before the row's data, so that
    every block boundary after the first shifts."""
    def bad(x):
        rows, k = x.shape
        kp = -(-k // O.BLOCK) * O.BLOCK
        if kp == k:
            return x
        out = np.zeros((rows, kp), dtype=x.dtype)
        out[:, kp - k:] = x
        return out
    monkeypatch.setattr(O, "pad_final_block", bad)
    assert caught(lambda: T.test_partial_final_block_worked_example(),
                  lambda: T.test_ragged_k_gemm_of_lossless_integers_is_the_integer_matmul(48))
