"""Back-to-back weight-streaming calls on one stream.

The streaming kernels are launched with programmatic dependent launch: a
call may start streaming its weights while the previous call on the stream
finishes, and waits for it before reading activations or writing outputs.
Here layer 2 consumes layer 1's output on the same stream; the chained
result must equal (bit for bit) the result with a synchronisation between
the calls, both eagerly and inside a CUDA graph. Both layers are checked
against the oracle: layer 1 on x, and layer 2 (whose griddepcontrol.wait is
the one that gates on a predecessor) on the bf16 output of layer 1.
"""
import pytest
import torch

import oracle
import synth
from gpu_cases import assert_within, bf16_to_f64, lib

pytestmark = pytest.mark.gpu


def _layers():
    mx = lib()
    w1 = synth.weights(21, 1024, 2048, device="cuda")
    w2 = synth.weights(22, 3072, 1024, device="cuda")
    q1, s1 = mx.quantize(w1)
    q2, s2 = mx.quantize(w2)
    x = synth.tokens(21, 4, 2048, device="cuda")
    return mx, (q1, s1), (q2, s2), x, w1, w2


def test_chained_layers_match_serialized():
    mx, (q1, s1), (q2, s2), x, w1, w2 = _layers()
    y1 = mx.linear(x, q1, s1)
    y2 = mx.linear(y1, q2, s2)  # no synchronisation between the calls
    torch.cuda.synchronize()
    y1s = mx.linear(x, q1, s1)
    torch.cuda.synchronize()
    y2s = mx.linear(y1s, q2, s2)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y1s.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), y2s.view(torch.int16))
    rq, rs = oracle.quantize(w1.cpu().numpy())
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y1), y_ref, rss, "layer 1")
    rq2, rs2 = oracle.quantize(w2.cpu().numpy())
    y2_ref, rss2 = oracle.linear(y1, rq2, rs2)  # the chained call against its own input
    assert_within(bf16_to_f64(y2), y2_ref, rss2, "layer 2 (chained)")
    assert mx.last_device_status() == mx.MXFP4_OK


def test_chained_layers_in_cuda_graph():
    mx, (q1, s1), (q2, s2), x, _, w2 = _layers()
    y1 = torch.empty((4, 1024), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((4, 3072), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mx.linear(x, q1, s1, out=y1)  # first calls outside the capture set per-device state
        mx.linear(y1, q2, s2, out=y2)
    s.synchronize()
    ref = y2.clone()
    y2.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.linear(x, q1, s1, out=y1)
        mx.linear(y1, q2, s2, out=y2)
    for _ in range(3):
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y2.view(torch.int16), ref.view(torch.int16))
    rq2, rs2 = oracle.quantize(w2.cpu().numpy())
    y2_ref, rss2 = oracle.linear(y1, rq2, rs2)
    assert_within(bf16_to_f64(y2), y2_ref, rss2, "layer 2 (graph)")
