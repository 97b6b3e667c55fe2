"""GPU parity of the fused dense FFN chain (mxfp4_ffn: up -> SwiGLU -> down
in one cooperative launch) against the oracle's SwiGLU FFN (the one-expert
MoE), within the stated bound; output and workspace between guard bytes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_cases import Guarded, assert_within, bf16_to_f64, lib

pytestmark = pytest.mark.gpu


def _weights(seed, hidden, inter):
    mx = lib()
    w1 = synth.weights(seed, 2 * inter, hidden, device="cuda")
    w2 = synth.weights(seed, hidden, inter, tid=synth.TID_W2, device="cuda")
    w1q, w1s = mx.quantize(w1)
    w2q, w2s = mx.quantize(w2)
    return (w1q, w1s, w2q, w2s), (w1, w2)


def _run(x, dev):
    mx = lib()
    t, hidden = x.shape
    inter = dev[2].shape[1] * 2
    y = Guarded((t, hidden), torch.bfloat16)
    ws = Guarded((mx.mxfp4_ffn_workspace_size(t, hidden, inter),), torch.uint8)
    mx.ffn(x, *dev, workspace=ws.t, out=y.t)
    for buf, name in ((y, "y"), (ws, "workspace")):
        buf.check(f"ffn t={t} hidden={hidden} inter={inter}: {name}")
    assert mx.last_device_status() == mx.MXFP4_OK
    return y.t


@pytest.mark.parametrize("t,hidden,inter", [(1, 256, 128), (4, 512, 256), (5, 256, 384), (8, 1024, 512),
                                            (3, 96, 160), (2, 2048, 1024), (8, 4096, 1536), (6, 7168, 512),
                                            (3, 1024, 1536), (1, 512, 512), (4, 7168, 512), (2, 1536, 7168)])
def test_ffn_small(t, hidden, inter):
    """The two-launch packed-E2M1 chain where t <= 4 and hidden, inter are
    multiples of 512 (t = 3: padding rows of the MMA's N; hidden = 512: one
    stage for the up projection; inter = 512: one stage for the down one),
    the cooperative kernel otherwise."""
    seed = 900 + t + hidden + inter
    dev, _ = _weights(seed, hidden, inter)
    x = synth.tokens(seed, t, hidden, device="cuda")
    y = _run(x, dev)
    q = [a.cpu().numpy() for a in dev]
    y_ref, rss = oracle.ffn(x, *q, inter)
    assert_within(bf16_to_f64(y), y_ref, rss, f"ffn t={t} hidden={hidden} inter={inter}")


def test_ffn_matches_linear_composition():
    """The same chain from the library's own parts: mxfp4_linear for W1,
    SwiGLU in float64 on the host, then the oracle's linear for W2. Checks
    the gate / up row order and the hand-off between the phases."""
    mx = lib()
    t, hidden, inter = 4, 1024, 512
    dev, _ = _weights(77, hidden, inter)
    x = synth.tokens(77, t, hidden, device="cuda")
    y = _run(x, dev)
    w1q, w1s, w2q, w2s = (a.cpu().numpy() for a in dev)
    ab, _ = oracle.linear(x, w1q, w1s)  # [t, 2*inter] float64
    a, b = ab[:, :inter], ab[:, inter:]
    h = a / (1.0 + np.exp(-a)) * b
    dec2 = oracle.dequant(w2q, w2s)
    ref = h @ dec2.T
    rss = np.sqrt((h ** 2) @ (dec2 ** 2).T)
    assert_within(bf16_to_f64(y), ref, rss, "ffn vs linear composition")


def test_ffn_deterministic():
    t, hidden, inter = 8, 2048, 1024
    dev, _ = _weights(5, hidden, inter)
    x = synth.tokens(5, t, hidden, device="cuda")
    y1 = _run(x, dev)
    y2 = _run(x, dev)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("t,inter", [(1, 9216), (4, 9216), (8, 2048)])
def test_ffn_full_size_sampled(t, inter):
    """hidden 7168 with the FFN width of the bench (inter 9216: W1 [18432,
    7168], W2 [7168, 9216]) and with an expert-sized inter 2048 at t = 8;
    512 sampled output columns per token against the oracle."""
    hidden = 7168
    dev, _ = _weights(11, hidden, inter)
    x = synth.tokens(11 + t, t, hidden, device="cuda")
    y = _run(x, dev)
    cols = np.sort(np.random.default_rng(t).choice(hidden, 512, replace=False))
    q = [a.cpu().numpy() for a in dev]
    y_ref, rss = oracle.ffn(x, *q, inter, cols=cols)
    assert_within(bf16_to_f64(y)[:, cols], y_ref, rss, f"ffn full size t={t} inter={inter}")


def test_ffn_shape_that_does_not_fit():
    """t = 5 at inter 9216: the down phase's staged h (2t columns of all of
    K) does not fit on chip, so the call refuses before any launch."""
    mx = lib()
    t, hidden, inter = 5, 7168, 9216
    x = torch.zeros((t, hidden), dtype=torch.bfloat16, device="cuda")
    w1q = torch.zeros((2 * inter, hidden // 2), dtype=torch.uint8, device="cuda")
    w1s = torch.zeros((2 * inter, hidden // 32), dtype=torch.uint8, device="cuda")
    w2q = torch.zeros((hidden, inter // 2), dtype=torch.uint8, device="cuda")
    w2s = torch.zeros((hidden, inter // 32), dtype=torch.uint8, device="cuda")
    y = torch.zeros((t, hidden), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(mx.mxfp4_ffn_workspace_size(t, hidden, inter), dtype=torch.uint8, device="cuda")
    rc = mx.mxfp4_ffn(x.data_ptr(), t, hidden, w1q.data_ptr(), w1s.data_ptr(), w2q.data_ptr(), w2s.data_ptr(),
                      inter, y.data_ptr(), ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == mx.MXFP4_ERR_SHAPE
    assert int(ws.sum()) == 0 and int(y.view(torch.int16).abs().sum()) == 0  # nothing was launched
