"""GPU parity of mxfp4_moe against the oracle: routing indices bit-exact,
gate weights within 1e-6 relative, outputs within the stated bound (the RSS
term runs over every (expert, j) term g_e * h_ej * w2_ej)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_cases import assert_within, bf16_to_f64, lib

pytestmark = pytest.mark.gpu


def _experts(seed, e, hidden, inter, device="cuda"):
    """Packed expert weights on the device plus host packings from the oracle."""
    mx = lib()
    w1 = synth.weights(seed, e * 2 * inter, hidden, device=device)
    w2 = synth.weights(seed, e * hidden, inter, tid=synth.TID_W2, device=device)
    w1q, w1s = mx.quantize(w1)
    w2q, w2s = mx.quantize(w2)
    r1q, r1s = oracle.quantize(w1.cpu().numpy())
    r2q, r2s = oracle.quantize(w2.cpu().numpy())
    assert np.array_equal(w1q.cpu().numpy(), r1q) and np.array_equal(w2q.cpu().numpy(), r2q)
    W1 = {ex: (r1q.reshape(e, 2 * inter, -1)[ex], r1s.reshape(e, 2 * inter, -1)[ex]) for ex in range(e)}
    W2 = {ex: (r2q.reshape(e, hidden, -1)[ex], r2s.reshape(e, hidden, -1)[ex]) for ex in range(e)}
    dev = (w1q.view(e, 2 * inter, hidden // 2), w1s.view(e, 2 * inter, hidden // 32),
           w2q.view(e, hidden, inter // 2), w2s.view(e, hidden, inter // 32))
    return dev, W1, W2


def _run(x, lg, top_k, dev):
    mx = lib()
    t = x.shape[0]
    ids = torch.empty((t, top_k), dtype=torch.int32, device="cuda")
    gw = torch.empty((t, top_k), dtype=torch.float32, device="cuda")
    y = mx.moe(x, lg, top_k, *dev, topk_ids=ids, topk_w=gw)
    torch.cuda.synchronize()
    return y, ids, gw


@pytest.mark.parametrize("t,e,top_k,hidden,inter", [(8, 16, 4, 256, 128), (32, 64, 8, 512, 256), (1, 8, 1, 64, 32),
                                                    (5, 12, 3, 96, 160), (32, 8, 8, 128, 64)])
def test_moe_small(t, e, top_k, hidden, inter):
    seed = t + e
    dev, W1, W2 = _experts(seed, e, hidden, inter)
    x = synth.tokens(seed, t, hidden, device="cuda")
    lg = synth.logits(seed, t, e, device="cuda")
    y, ids, gw = _run(x, lg, top_k, dev)
    lgn = lg.cpu().numpy()
    ids_ref, g_ref = oracle.route(lgn, top_k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.allclose(gw.cpu().numpy(), g_ref, rtol=1e-6, atol=0)
    y_ref, rss = oracle.moe(x, lgn, top_k, W1, W2, inter)
    assert_within(bf16_to_f64(y), y_ref, rss, f"moe t={t} e={e} k={top_k}")


def test_moe_routing_ties_and_hot_expert():
    """Equal logits (ties to smaller index) and every token on the same
    experts: one expert gets all 32 tokens (several chunks)."""
    t, e, top_k, hidden, inter = 32, 16, 4, 128, 64
    dev, W1, W2 = _experts(77, e, hidden, inter)
    x = synth.tokens(77, t, hidden, device="cuda")
    lg = torch.zeros((t, e), dtype=torch.float32)
    lg[:, 5] = 3.0
    lg[::2, 9] = 3.0  # ties with expert 5 on even tokens -> 5 first
    lg = lg.cuda()
    y, ids, gw = _run(x, lg, top_k, dev)
    lgn = lg.cpu().numpy()
    ids_ref, g_ref = oracle.route(lgn, top_k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.allclose(gw.cpu().numpy(), g_ref, rtol=1e-6, atol=0)
    y_ref, rss = oracle.moe(x, lgn, top_k, W1, W2, inter)
    assert_within(bf16_to_f64(y), y_ref, rss, "moe hot expert")


def test_moe_deterministic_and_status():
    mx = lib()
    t, e, top_k, hidden, inter = 16, 32, 8, 256, 128
    dev, _, _ = _experts(3, e, hidden, inter)
    x = synth.tokens(3, t, hidden, device="cuda")
    lg = synth.logits(3, t, e, device="cuda")
    y1, _, _ = _run(x, lg, top_k, dev)
    y2, _, _ = _run(x, lg, top_k, dev)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert mx.last_device_status() == mx.MXFP4_OK


def test_moe_full_size_sampled():
    """256 experts, W1 [4096,7168], W2 [7168,2048], T=32, top-8: routing of all
    tokens bit-exact; sampled tokens x sampled outputs within tolerance. The
    oracle's packings of the experts those tokens use come from the same
    float32 weights the GPU packed."""
    mx = lib()
    t, e, top_k, hidden, inter, seed = 32, 256, 8, 7168, 2048, 4
    w1q = torch.empty((e, 2 * inter, hidden // 2), dtype=torch.uint8, device="cuda")
    w1s = torch.empty((e, 2 * inter, hidden // 32), dtype=torch.uint8, device="cuda")
    w2q = torch.empty((e, hidden, inter // 2), dtype=torch.uint8, device="cuda")
    w2s = torch.empty((e, hidden, inter // 32), dtype=torch.uint8, device="cuda")
    for ex in range(e):  # generate and pack one expert at a time
        a = synth.weights(seed, 2 * inter, hidden, device="cuda", row0=ex * 2 * inter)
        q, s = mx.quantize(a)
        w1q[ex].copy_(q.view(2 * inter, -1))
        w1s[ex].copy_(s.view(2 * inter, -1))
        b = synth.weights(seed, hidden, inter, tid=synth.TID_W2, device="cuda", row0=ex * hidden)
        q, s = mx.quantize(b)
        w2q[ex].copy_(q.view(hidden, -1))
        w2s[ex].copy_(s.view(hidden, -1))
    x = synth.tokens(seed, t, hidden, device="cuda")
    lg = synth.logits(seed, t, e, device="cuda")
    y, ids, gw = _run(x, lg, top_k, (w1q, w1s, w2q, w2s))
    lgn = lg.cpu().numpy()
    ids_ref, g_ref = oracle.route(lgn, top_k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.allclose(gw.cpu().numpy(), g_ref, rtol=1e-6, atol=0)
    toks = np.array([0, 13, 31])
    cols = np.random.default_rng(0).choice(hidden, 96, replace=False)
    need = sorted({int(v) for v in ids_ref[toks].ravel()})
    W1, W2 = {}, {}
    for ex in need:
        a = synth.weights(seed, 2 * inter, hidden, device="cuda", row0=ex * 2 * inter).cpu().numpy()
        W1[ex] = oracle.quantize(a)
        assert np.array_equal(W1[ex][0], w1q[ex].cpu().numpy())
        b = synth.weights(seed, hidden, inter, tid=synth.TID_W2, device="cuda", row0=ex * hidden).cpu().numpy()
        W2[ex] = oracle.quantize(b)
    y_ref, rss = oracle.moe(x, lgn, top_k, W1, W2, inter, tok=toks, cols=cols)
    yg = bf16_to_f64(y)[toks][:, cols]
    assert_within(yg, y_ref, rss, "moe full size")
