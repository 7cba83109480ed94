"""The C ABI's device-memory rule and its thread safety, through ctypes with
raw pointers: every entry point refuses a pointer that is not device memory
of the current GPU (host memory, pinned or not, reaches the GPU only
through unified addressing) before anything is launched, and the first
calls of several host threads at once set up the kernels without a race."""
import os
import subprocess
import sys

import pytest
import torch

from mxcheck import ROOT, ensure_built

pytestmark = pytest.mark.gpu

INVALID_ARG = 1


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def h():
    return int(torch.cuda.current_stream().cuda_stream)


def test_quantize_refuses_host_memory(mx):
    rows, cols = 128, 128
    x = torch.randn(rows, cols).to(torch.bfloat16)
    q = torch.full((rows, cols), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((mx.mx_scale_bytes(rows, cols),), 0xAB, dtype=torch.uint8, device="cuda")
    for host_x in (x, x.pin_memory()):          # pageable, then pinned (mapped) host memory
        assert mx.mx_quantize(host_x.data_ptr(), 0, rows, cols, cols, 0, 1, 0, q.data_ptr(),
                              s.data_ptr(), None, None, h()) == INVALID_ARG
    xd = x.cuda()
    hq = torch.empty((rows, cols), dtype=torch.uint8).pin_memory()
    assert mx.mx_quantize(xd.data_ptr(), 0, rows, cols, cols, 0, 1, 0, hq.data_ptr(),
                          s.data_ptr(), None, None, h()) == INVALID_ARG
    rb = torch.zeros(rows, cols, dtype=torch.int16).pin_memory()
    assert mx.mx_quantize_sr(xd.data_ptr(), 0, rows, cols, cols, rb.data_ptr(), cols, 0, 1, 0,
                             q.data_ptr(), s.data_ptr(), None, None, h()) == INVALID_ARG
    torch.cuda.synchronize()
    assert (q == 0xAB).all() and (s == 0xAB).all()      # nothing was launched
    assert mx.mx_device_status(h()) == 0


def test_gemms_refuse_host_memory(mx):
    m = n = k = 128
    qa = mx.quantize(torch.randn(m, k).to(torch.bfloat16).cuda(), "e4m3", "row")
    qb = mx.quantize(torch.randn(k, n).to(torch.bfloat16).cuda(), "e4m3", "col")
    y = torch.full((m, n), 7.0, device="cuda")
    hy = torch.empty(m, n).pin_memory()
    ha = qa.codes.cpu().pin_memory()
    assert mx.mx_gemm(m, n, k, qa.codes.data_ptr(), qa.scales.data_ptr(), 0, qb.codes.data_ptr(),
                      qb.scales.data_ptr(), 0, hy.data_ptr(), 1, n, h()) == INVALID_ARG
    assert mx.mx_gemm(m, n, k, ha.data_ptr(), qa.scales.data_ptr(), 0, qb.codes.data_ptr(),
                      qb.scales.data_ptr(), 0, y.data_ptr(), 1, n, h()) == INVALID_ARG
    bias = torch.zeros(n).pin_memory()
    assert mx.mx_gemm_bias_act(m, n, k, qa.codes.data_ptr(), qa.scales.data_ptr(), 0,
                               qb.codes.data_ptr(), qb.scales.data_ptr(), 0, bias.data_ptr(), 1,
                               y.data_ptr(), 1, n, h()) == INVALID_ARG
    # group offsets in host memory
    off = torch.tensor([0, m], dtype=torch.int32).pin_memory()
    assert mx.mx_grouped_gemm(1, off.data_ptr(), m, n, k, qa.codes.data_ptr(),
                              qa.scales.data_ptr(), 0, qb.codes.data_ptr(), qb.scales.data_ptr(),
                              0, y.data_ptr(), 1, h()) == INVALID_ARG
    torch.cuda.synchronize()
    assert (y == 7.0).all()
    # the same call with device memory everywhere runs
    assert mx.mx_gemm(m, n, k, qa.codes.data_ptr(), qa.scales.data_ptr(), 0, qb.codes.data_ptr(),
                      qb.scales.data_ptr(), 0, y.data_ptr(), 1, n, h()) == 0
    assert mx.mx_device_status(h()) == 0


def test_tensor_api_refuses_host_tensors(mx):
    x = torch.randn(64, 64).to(torch.bfloat16)
    with pytest.raises(ValueError):
        mx.quantize(x, "e4m3", "row")
    qa = mx.quantize(x.cuda(), "e4m3", "row")
    qb = mx.quantize(x.cuda(), "e4m3", "col")
    with pytest.raises(ValueError):
        mx.gemm(qa, qb, "fp32", out=torch.empty(64, 64))
    with pytest.raises(ValueError):
        mx.gemm(qa, qb, "fp32", bias=torch.zeros(64))


FIRST_CALLS = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import mxfp8_block_scaled_mx_gb300 as mx
torch.cuda.init()
m, n, k = 256, 512, 256
g = torch.Generator().manual_seed(0)
x = torch.randn(m, k, generator=g).to(torch.bfloat16).cuda()
w = torch.randn(k, n, generator=g).to(torch.bfloat16).cuda()
streams = [torch.cuda.Stream() for _ in range(4)]
outs = [None] * 4
errors = []

def run(i):
    try:
        torch.cuda.set_device(0)
        with torch.cuda.stream(streams[i]):
            qa = mx.quantize(x, "e4m3", "row", stream=streams[i])
            qb = mx.quantize(w, "e4m3", "col", stream=streams[i])
            outs[i] = mx.gemm(qa, qb, "fp32", stream=streams[i])
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=run, args=(i,)) for i in range(4)]
for t in threads:
    t.start()
for t in threads:
    t.join()
torch.cuda.synchronize()
assert not errors, errors
for o in outs[1:]:
    assert torch.equal(o, outs[0])
assert mx.device_status() == 0
print("ok")
"""


def test_first_calls_from_several_threads(mx):
    """Four host threads make the library's first quantize and GEMM calls
    of a fresh process at the same time, each on its own stream: the
    per-device set-up runs once, and all four results agree exactly."""
    res = subprocess.run([sys.executable, "-c", FIRST_CALLS, ROOT], capture_output=True,
                         text=True, timeout=300, env=dict(os.environ))
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip().endswith("ok")
