"""Host-only checks of the C ABI (no GPU): the library loads, exports every
symbol include/mx.h declares, computes buffer sizes, and rejects invalid
arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

from mxcheck import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "mx.h")


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mx_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(mx):
    names = declared_functions()
    assert len(names) >= 10
    handle = ctypes.CDLL(mx.LIB_PATH)
    for name in names:
        assert hasattr(handle, name), name
    assert set(names) == set(mx.EXPORTS)


def test_scale_bytes(mx):
    assert mx.mx_scale_bytes(256, 512) == 256 * 16
    assert mx.mx_scale_bytes(1, 32) == 128 * 4
    assert mx.mx_scale_bytes(130, 160) == 256 * 8
    assert mx.mx_scale_bytes(16384, 7168) == 16384 * 224
    assert mx.mx_scale_bytes(10, 33) == 0
    assert mx.mx_scale_bytes(10, 40) == 0                 # k % 16
    assert mx.mx_scale_bytes(130, 48) == 256 * 4          # a partial final block of 16
    assert mx.mx_scale_bytes(1, 16) == 128 * 4
    assert mx.mx_grouped_scale_bytes(65536, 64, 7168) == (512 + 64) * 128 * 224
    assert mx.mx_status_str(0) == "MX_OK"
    assert mx.mx_status_str(5) == "MX_ERR_TIMEOUT"


FAKE = 0x10000  # an aligned non-null address; validation rejects before any use


def test_quantize_rejects_bad_arguments_on_the_host(mx):
    q = mx.mx_quantize
    s = 0
    # K (cols) not a multiple of 16 for rowwise
    assert q(FAKE, 0, 64, 40, 40, 0, 1, 0, FAKE, FAKE, None, None, s) == 1
    # rows not a multiple of 16 for colwise
    assert q(FAKE, 0, 40, 64, 64, 0, 2, 0, None, None, FAKE, FAKE, s) == 1
    # packed storage: the blocked axis in whole 32-element blocks
    assert q(FAKE, 0, 64, 48, 48, 7, 1, 0, FAKE, FAKE, None, None, s) == 1
    assert q(FAKE, 0, 48, 64, 64, 5, 2, 0, None, None, FAKE, FAKE, s) == 1
    # bad enums
    assert q(FAKE, 0, 64, 64, 64, 8, 1, 0, FAKE, FAKE, None, None, s) == 1
    assert q(FAKE, 0, 64, 64, 64, 0, 4, 0, FAKE, FAKE, None, None, s) == 1
    assert q(FAKE, 0, 64, 64, 64, 0, 1, 9, FAKE, FAKE, None, None, s) == 1
    # input types: bf16 (0) and fp32 (1) only
    assert q(FAKE, 2, 64, 64, 64, 0, 1, 0, FAKE, FAKE, None, None, s) == 1
    # fp32 rows must start on 16-byte boundaries: ldx % 4
    assert q(FAKE, 1, 64, 64, 66, 0, 1, 0, FAKE, FAKE, None, None, s) == 2
    # fp32 tiles are 64 columns wide: 3 * 2^24 row tiles x 128 column tiles
    # are 2^32 or more (as bf16, 64 column tiles, they would fit)
    assert q(FAKE, 1, 3 << 31, 8192, 8192, 0, 1, 0, FAKE, FAKE, None, None, s) == 3
    # null outputs
    assert q(FAKE, 0, 64, 64, 64, 0, 1, 0, None, FAKE, None, None, s) == 1
    assert q(None, 0, 64, 64, 64, 0, 1, 0, FAKE, FAKE, None, None, s) == 1
    # ldx < cols
    assert q(FAKE, 0, 64, 64, 32, 0, 1, 0, FAKE, FAKE, None, None, s) == 1
    # misaligned input pointer / leading dimension
    assert q(FAKE + 2, 0, 64, 64, 64, 0, 1, 0, FAKE, FAKE, None, None, s) == 2
    assert q(FAKE, 0, 64, 64, 68, 0, 1, 0, FAKE, FAKE, None, None, s) == 2
    assert q(FAKE, 0, 64, 64, 64, 0, 1, 0, FAKE + 8, FAKE, None, None, s) == 2
    # 2^32 or more 128x128 tiles (tile numbers are 32-bit)
    assert q(FAKE, 0, 1 << 40, 8192, 8192, 0, 1, 0, FAKE, FAKE, None, None, s) == 3


def test_gemm_rejects_bad_arguments_on_the_host(mx):
    g = mx.mx_gemm
    s = 0
    ok = dict(m=64, n=64, k=64)
    assert g(64, 64, 40, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 64, s) == 1      # k % 16
    assert g(64, 64, 48, FAKE, FAKE, 7, FAKE, FAKE, 0, FAKE, 0, 64, s) == 1      # packed: k % 128
    assert g(64, 64, 0, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 64, s) == 1       # k == 0
    assert g(64, 60, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 64, s) == 1      # n % 8
    assert g(64, 64, 64, FAKE, FAKE, 7, FAKE, FAKE, 0, FAKE, 0, 64, s) == 1      # fmt
    assert g(64, 64, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 5, 64, s) == 1      # out dtype
    assert g(64, 64, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 32, s) == 1      # ldy < n
    assert g(64, 64, 64, None, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 64, s) == 1      # null
    assert g(64, 64, 64, FAKE + 4, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 64, s) == 2  # misaligned
    assert g(64, 64, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 68, s) == 2      # ldy*2 % 16
    big = 1 << 30                                       # 2^44 work units: beyond 32-bit indexing
    assert g(big, big, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, big, s) == 3
    assert ok


def test_grouped_calls_reject_bad_arguments_on_the_host(mx):
    gg = mx.mx_grouped_gemm
    assert gg(0, FAKE, 64, 128, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 0) == 1      # groups
    assert gg(2000, FAKE, 64, 128, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 0) == 1   # > 1000
    assert gg(4, None, 64, 128, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 0) == 1      # offsets
    assert gg(4, FAKE, 64, 136, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 0, 0) == 1      # n % 128
    qg = mx.mx_quantize_grouped
    assert qg(FAKE, 0, 64, 64, 64, 0, 0, 0, FAKE, FAKE, FAKE, 0) == 1                  # groups
    assert qg(FAKE, 0, 64, 40, 40, 0, 0, 4, FAKE, FAKE, FAKE, 0) == 1                  # cols % 16
    assert qg(FAKE, 0, 64, 64, 64, 0, 0, 4, None, FAKE, FAKE, 0) == 1                  # offsets


def test_grouped_backward_calls_reject_bad_arguments_on_the_host(mx):
    assert mx.mx_grouped_cols_capacity(65536, 64) == (512 + 64) * 128
    assert mx.mx_grouped_cols_capacity(200, 7) == (1 + 7) * 128
    assert mx.mx_grouped_cols_capacity(-1, 4) == 0
    qx = mx.mx_quantize_grouped_ex
    # (x, dtype, total, cols, ldx, fmt, axis, rule, groups, offsets, q_row, s_row, q_col, ldq, s_col, s)
    assert qx(FAKE, 0, 64, 64, 64, 0, 2, 0, 4, FAKE, None, None, FAKE, 200, FAKE, 0) == 1   # ldq % 128
    assert qx(FAKE, 0, 64, 64, 64, 0, 2, 0, 4, FAKE, None, None, FAKE, 0, FAKE, 0) == 1     # ldq == 0
    assert qx(FAKE, 0, 64, 64, 64, 0, 2, 0, 4, FAKE, None, None, None, 256, FAKE, 0) == 1  # q_col
    assert qx(FAKE, 0, 64, 64, 64, 0, 2, 0, 4, None, None, None, FAKE, 256, FAKE, 0) == 1  # offsets
    assert qx(FAKE, 0, 64, 64, 64, 0, 2, 0, 0, FAKE, None, None, FAKE, 256, FAKE, 0) == 1  # groups
    assert qx(FAKE, 0, 64, 40, 40, 0, 3, 0, 4, FAKE, FAKE, FAKE, FAKE, 256, FAKE, 0) == 1  # row cols % 16
    assert qx(FAKE, 0, 64, 64, 64, 0, 2, 0, 4, FAKE, None, None, FAKE + 8, 256, FAKE, 0) == 2  # align
    # (2^24 + 4) x 65535 padded column tiles: beyond 32-bit tile numbers
    big = (1 << 31) - 1
    assert qx(FAKE, 0, big, 65535 * 128, 65535 * 128, 0, 2, 0, 4, FAKE, None, None, FAKE,
              1 << 31, FAKE, 0) == 3
    bc = mx.mx_grouped_gemm_bcat
    # (groups, offsets, total_m, n, k, a, sa, fa, b, ldb, sb, fb, y, y_dtype, s)
    assert bc(4, FAKE, 64, 128, 96, FAKE, FAKE, 0, FAKE, 384, FAKE, 0, FAKE, 0, 0) == 1     # k % 128
    assert bc(4, FAKE, 64, 128, 128, FAKE, FAKE, 0, FAKE, 384, FAKE, 0, FAKE, 0, 0) == 1    # ldb < g*k
    assert bc(4, None, 64, 128, 128, FAKE, FAKE, 0, FAKE, 512, FAKE, 0, FAKE, 0, 0) == 1    # offsets
    assert bc(4, FAKE, 64, 128, 128, FAKE, FAKE, 0, FAKE, 520, FAKE, 0, FAKE, 0, 0) == 2    # ldb % 16
    wg = mx.mx_grouped_gemm_wgrad
    # (groups, offsets, total, m, n, ldk, a, sa, fa, b, sb, fb, y, y_dtype, s)
    assert wg(4, FAKE, 100, 64, 64, 200, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 1, 0) == 1      # ldk % 128
    assert wg(4, FAKE, -1, 64, 64, 256, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 1, 0) == 1       # total
    assert wg(0, FAKE, 100, 64, 64, 256, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 1, 0) == 1      # groups
    assert wg(4, FAKE, 100, 64, 60, 256, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 1, 0) == 1      # n % 8
    assert wg(4, FAKE, 100, 64, 64, 256, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE + 4, 1, 0) == 2  # y align
    # 1000 experts x 4096 x 4096 work units of 256x256: more than 2^31
    assert wg(1000, FAKE, 100, 1 << 20, 1 << 20, 256, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 1, 0) == 3


def test_fused_epilogue_rejects_bad_arguments_on_the_host(mx):
    f = mx.mx_gemm_bias_act
    assert f(64, 64, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, None, 7, FAKE, 0, 64, 0) == 1      # act
    assert f(64, 64, 64, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE + 4, 1, FAKE, 0, 64, 0) == 2  # bias align
    assert f(64, 64, 40, FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 1, FAKE, 0, 64, 0) == 1      # k % 16


def test_stochastic_quantize_rejects_bad_arguments_on_the_host(mx):
    q = mx.mx_quantize_sr
    assert q(FAKE, 0, 64, 64, 64, None, 64, 0, 1, 0, FAKE, FAKE, None, None, 0) == 1     # no rbits
    assert q(FAKE, 0, 64, 64, 64, FAKE, 32, 0, 1, 0, FAKE, FAKE, None, None, 0) == 1     # ldr < cols
    assert q(FAKE, 0, 64, 64, 64, FAKE + 2, 64, 0, 1, 0, FAKE, FAKE, None, None, 0) == 2  # align
    assert q(FAKE, 0, 64, 64, 64, FAKE, 68, 0, 1, 0, FAKE, FAKE, None, None, 0) == 2     # ldr % 8


def test_narrow_formats_on_the_host(mx):
    """MXFP6 / MXFP4 codes: accepted by the quantizer, stochastic rounding
    and the GEMM (the host checks apply as for FP8); not by the grouped
    quantizer (FP8 only)."""
    sr = mx.mx_quantize_sr
    for fmt in (2, 3, 4):
        assert sr(FAKE, 0, 64, 64, 64, FAKE, 64, fmt, 1, 0, FAKE, FAKE, None, None, 0) != 3
        assert sr(FAKE, 0, 64, 64, 64, FAKE, 32, fmt, 1, 0, FAKE, FAKE, None, None, 0) == 1
        assert sr(FAKE, 0, 64, 64, 64, FAKE + 2, 64, fmt, 1, 0, FAKE, FAKE, None, None, 0) == 2
        assert mx.mx_quantize_grouped(FAKE, 0, 64, 64, 64, fmt, 0, 4, FAKE, FAKE, FAKE, 0) == 3
    q = mx.mx_quantize
    assert q(FAKE, 0, 64, 64, 64, 8, 1, 0, FAKE, FAKE, None, None, 0) == 1           # no format 8
    assert q(FAKE, 0, 64, 40, 40, 4, 1, 0, FAKE, FAKE, None, None, 0) == 1           # cols % 16


def test_packed_formats_on_the_host(mx):
    """Packed 6- and 4-bit storage (formats 5-7): the GEMM wants K % 128 and
    32-byte aligned packed code pointers; stochastic rounding accepts them,
    the grouped quantizer stays FP8 only."""
    g = mx.mx_gemm
    for fmt in (5, 6, 7):
        assert g(64, 64, 96, FAKE, FAKE, fmt, FAKE, FAKE, 0, FAKE, 0, 64, 0) == 1        # k % 128
        assert g(64, 64, 96, FAKE, FAKE, 0, FAKE, FAKE, fmt, FAKE, 0, 64, 0) == 1
        assert g(64, 64, 128, FAKE + 16, FAKE, fmt, FAKE, FAKE, 0, FAKE, 0, 64, 0) == 2  # a % 32
        assert g(64, 64, 128, FAKE, FAKE, 0, FAKE + 16, FAKE, fmt, FAKE, 0, 64, 0) == 2  # b % 32
        assert mx.mx_quantize_sr(FAKE, 0, 64, 64, 64, FAKE, 64, fmt, 1, 0, FAKE, FAKE, None, None,
                                 0) != 3
        assert mx.mx_quantize_grouped(FAKE, 0, 64, 64, 64, fmt, 0, 4, FAKE, FAKE, FAKE, 0) == 3
    assert mx.storage_bytes("e2m1_packed", 128) == 64
    assert mx.storage_bytes("e3m2_packed", 128) == 96
    assert mx.storage_bytes("e2m1", 128) == 128
    assert mx.storage_elems("e2m3_packed", 96) == 128


def test_selftest_rejects_zero_limit(mx):
    assert mx.mx_selftest_wait_timeout(0, 0) == 1


def test_no_cpu_fallback(monkeypatch):
    """Without the built library every entry point raises, and the tensor
    API refuses CPU tensors instead of computing anything on the host."""
    import torch
    import mxfp8_block_scaled_mx_gb300 as mx
    monkeypatch.setattr(mx, "_lib", None)
    monkeypatch.setattr(mx, "LIB_PATH", os.path.join(ROOT, "no-such-libmx.so"))
    with pytest.raises(RuntimeError):
        mx.mx_scale_bytes(128, 128)
    with pytest.raises(RuntimeError):
        mx.device_status()
    x = torch.zeros(64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mx.quantize(x, "e4m3", "row")
    codes = torch.zeros(64, 64, dtype=torch.uint8)
    t = mx.MxTensor(codes, torch.zeros(1024, dtype=torch.uint8), "e4m3")
    with pytest.raises(ValueError):
        mx.gemm(t, t, "fp32")
    with pytest.raises(ValueError):
        mx.quantize_grouped(x, torch.tensor([0, 64], dtype=torch.int32))
