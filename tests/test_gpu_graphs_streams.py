"""The library inside CUDA graphs and on concurrent streams: it allocates no
device memory, keeps no per-call device scratch and never synchronizes, so
quantize + GEMM can be captured into a graph and replayed, and independent
calls on two streams may run at the same time."""
import pytest
import torch

from mxcheck import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    ensure_built()
    import mxfp8_block_scaled_mx_gb300 as mx
    return mx


def layer(seed, m=512, n=768, k=1024):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(m, k, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(k, n, generator=g) * 0.05).to(torch.bfloat16).cuda()
    return x, w


def test_quantize_and_gemm_captured_in_a_graph(mx):
    x, w = layer(1)
    eager = mx.gemm(mx.quantize(x, "e4m3", "row"), mx.quantize(w, "e4m3", "col"), "bf16")
    assert mx.device_status() == 0
    capture = torch.cuda.Stream()
    capture.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=capture):
        y = mx.gemm(mx.quantize(x, "e4m3", "row"), mx.quantize(w, "e4m3", "col"), "bf16")
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, eager)
    # new inputs written into the captured buffers are picked up on replay
    x2, w2 = layer(2)
    x.copy_(x2)
    w.copy_(w2)
    graph.replay()
    torch.cuda.synchronize()
    ref = mx.gemm(mx.quantize(x2, "e4m3", "row"), mx.quantize(w2, "e4m3", "col"), "bf16")
    assert torch.equal(y, ref)
    assert mx.device_status() == 0


def test_independent_calls_on_two_streams(mx):
    layers = [layer(s) for s in (3, 4)]
    seq = [mx.gemm(mx.quantize(x, "e4m3", "row"), mx.quantize(w, "e4m3", "col"), "fp32")
           for x, w in layers]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for (x, w), s in zip(layers, streams):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(4):
                y = mx.gemm(mx.quantize(x, "e4m3", "row"), mx.quantize(w, "e4m3", "col"), "fp32")
            outs.append(y)
    torch.cuda.synchronize()
    for got, ref in zip(outs, seq):
        assert torch.equal(got, ref)
    assert mx.device_status() == 0
