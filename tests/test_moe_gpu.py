"""GPU parity of mxfp4_moe against the oracle: routing indices bit-exact,
gate weights within 1e-6 relative, outputs within the stated bound (the RSS
term runs over every (expert, j) term g_e * h_ej * w2_ej)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_cases import Guarded, assert_within, bf16_to_f64, lib

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
    """One mxfp4_moe call whose outputs and workspace all sit between guard
    bytes; checks that nothing outside them was written."""
    mx = lib()
    t, hidden = x.shape
    e = lg.shape[1]
    inter = dev[2].shape[2] * 2
    ids = Guarded((t, top_k), torch.int32)
    gw = Guarded((t, top_k), torch.float32)
    y = Guarded((t, hidden), torch.bfloat16)
    ws = Guarded((mx.mxfp4_moe_workspace_size(t, e, top_k, hidden, inter),), torch.uint8)
    mx.moe(x, lg, top_k, *dev, workspace=ws.t, out=y.t, topk_ids=ids.t, topk_w=gw.t)
    for buf, name in ((ids, "topk_ids"), (gw, "topk_w"), (y, "y"), (ws, "workspace")):
        buf.check(f"moe t={t} e={e} top_k={top_k}: {name}")
    return y.t, ids.t, gw.t


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


@pytest.mark.parametrize("t,e,top_k,hidden,inter", [(64, 64, 8, 256, 128), (128, 128, 8, 256, 128),
                                                    (256, 128, 8, 256, 128), (256, 32, 16, 128, 64),
                                                    (64, 1024, 16, 128, 64)])
def test_moe_larger_t(t, e, top_k, hidden, inter):
    """Token counts up to the header's limit (t <= 256), and its largest e
    and top_k: many experts receive more tokens than one chunk holds."""
    seed = 1000 + t + e + top_k
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


@pytest.mark.parametrize("t,e,top_k,n_shared,hidden,inter", [(8, 16, 4, 1, 256, 128), (32, 64, 8, 2, 512, 256),
                                                             (1, 8, 1, 1, 64, 32), (256, 32, 8, 1, 128, 64)])
def test_moe_shared_experts(t, e, top_k, n_shared, hidden, inter):
    """mxfp4_moe_shared: the weight arrays hold e routed then n_shared shared
    experts; every token adds each shared expert's output with weight 1."""
    mx = lib()
    seed = 500 + t + e + n_shared
    dev, W1, W2 = _experts(seed, e + n_shared, hidden, inter)
    x = synth.tokens(seed, t, hidden, device="cuda")
    lg = synth.logits(seed, t, e, device="cuda")
    ids = Guarded((t, top_k), torch.int32)
    gw = Guarded((t, top_k), torch.float32)
    y = Guarded((t, hidden), torch.bfloat16)
    ws = Guarded((mx.mxfp4_moe_shared_workspace_size(t, e, top_k, n_shared, hidden, inter),), torch.uint8)
    mx.moe(x, lg, top_k, *dev, workspace=ws.t, out=y.t, topk_ids=ids.t, topk_w=gw.t, n_shared=n_shared)
    for buf, name in ((ids, "topk_ids"), (gw, "topk_w"), (y, "y"), (ws, "workspace")):
        buf.check(f"moe_shared t={t} e={e} n_shared={n_shared}: {name}")
    lgn = lg.cpu().numpy()
    ids_ref, g_ref = oracle.route(lgn, top_k)
    assert np.array_equal(ids.t.cpu().numpy(), ids_ref)
    assert np.allclose(gw.t.cpu().numpy(), g_ref, rtol=1e-6, atol=0)
    y_ref, rss = oracle.moe(x, lgn, top_k, W1, W2, inter, n_shared=n_shared)
    assert_within(bf16_to_f64(y.t), y_ref, rss, f"moe_shared t={t} e={e} n_shared={n_shared}")
    assert mx.last_device_status() == mx.MXFP4_OK


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


class FullSize:
    """256 experts, W1 [4096,7168], W2 [7168,2048] packed on the device (one
    expert generated and packed at a time), T=32 tokens, top-8."""
    t, e, top_k, hidden, inter, seed = 32, 256, 8, 7168, 2048, 4

    def __init__(self):
        mx = lib()
        t, e, hidden, inter, seed = self.t, self.e, self.hidden, self.inter, self.seed
        self.w1q = torch.empty((e, 2 * inter, hidden // 2), dtype=torch.uint8, device="cuda")
        self.w1s = torch.empty((e, 2 * inter, hidden // 32), dtype=torch.uint8, device="cuda")
        self.w2q = torch.empty((e, hidden, inter // 2), dtype=torch.uint8, device="cuda")
        self.w2s = torch.empty((e, hidden, inter // 32), dtype=torch.uint8, device="cuda")
        for ex in range(e):
            q, sc = mx.quantize(self.w1_float(ex))
            self.w1q[ex].copy_(q.view(2 * inter, -1))
            self.w1s[ex].copy_(sc.view(2 * inter, -1))
            q, sc = mx.quantize(self.w2_float(ex))
            self.w2q[ex].copy_(q.view(hidden, -1))
            self.w2s[ex].copy_(sc.view(hidden, -1))
        self.x = synth.tokens(seed, t, hidden, device="cuda")
        self.lg = synth.logits(seed, t, e, device="cuda")
        self.dev = (self.w1q, self.w1s, self.w2q, self.w2s)
        self.W1 = {}

    def w1_float(self, ex):
        return synth.weights(self.seed, 2 * self.inter, self.hidden, device="cuda", row0=ex * 2 * self.inter)

    def w2_float(self, ex):
        return synth.weights(self.seed, self.hidden, self.inter, tid=synth.TID_W2, device="cuda",
                             row0=ex * self.hidden)

    def oracle_weights(self, experts, cols):
        """Oracle packings, from the float32 weights, of every listed expert's
        W1 and of the W2 rows of the sampled output columns (the oracle reads
        no other W2 row; the rest of each array stays zero)."""
        W2 = {}
        for ex in experts:
            if ex not in self.W1:
                self.W1[ex] = oracle.quantize(self.w1_float(ex).cpu().numpy())
            wq = np.zeros((self.hidden, self.inter // 2), np.uint8)
            ws = np.zeros((self.hidden, self.inter // 32), np.uint8)
            rows = self.w2_float(ex)[torch.from_numpy(cols).cuda()].cpu().numpy()
            wq[cols], ws[cols] = oracle.quantize(rows)
            W2[ex] = (wq, ws)
        return {ex: self.W1[ex] for ex in experts}, W2


@pytest.fixture(scope="module")
def full_size():
    return FullSize()


def _check_full_size(fs, lg, what, ncols=512):
    y, ids, gw = _run(fs.x, lg, fs.top_k, fs.dev)
    lgn = lg.cpu().numpy()
    ids_ref, g_ref = oracle.route(lgn, fs.top_k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.allclose(gw.cpu().numpy(), g_ref, rtol=1e-6, atol=0)
    cols = np.sort(np.random.default_rng(0).choice(fs.hidden, ncols, replace=False))
    experts = sorted({int(v) for v in ids_ref.ravel()})
    W1, W2 = fs.oracle_weights(experts, cols)
    for ex in experts[:4]:  # the device packing of a few routed experts, byte for byte
        assert np.array_equal(W1[ex][0], fs.w1q[ex].cpu().numpy())
        assert np.array_equal(W1[ex][1], fs.w1s[ex].cpu().numpy())
    y_ref, rss = oracle.moe(fs.x, lgn, fs.top_k, W1, W2, fs.inter, cols=cols)
    assert_within(bf16_to_f64(y)[:, cols], y_ref, rss, what)
    return ids_ref


def test_moe_full_size_all_tokens_sampled_columns(full_size):
    """The bench shape with its own seeded logits: routing of all 32 tokens
    bit-exact, gate weights to 1e-6, and every token's output at 512 sampled
    columns within the stated bound."""
    _check_full_size(full_size, full_size.lg, "moe full size")


def test_moe_full_size_hot_expert(full_size):
    """The bench shape with 12 tokens forced onto expert 37: its gate/up
    rows serve 12 token columns (two chunks of at most 8) and its down rows
    12 pairs (three chunks of at most 4), so the expert is streamed once per
    chunk at full size. Every token, 512 sampled columns."""
    lg = full_size.lg.clone()
    lg[:12, 37] += 8.0
    ids_ref = _check_full_size(full_size, lg, "moe full size, hot expert")
    assert int((ids_ref == 37).sum()) >= 12
