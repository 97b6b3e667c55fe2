"""GPU parity of mxfp4_quantize and mxfp4_linear against the oracle.

Packing is compared byte for byte; outputs elementwise under the stated
bound |y - y_ref| <= 4e-3*|y_ref| + 1e-3*sqrt(sum_k (x_k*w_k)^2).
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins
import synth
from gpu_cases import Guarded, assert_within, bf16_to_f64, lib, linear_case, sample_rows

pytestmark = pytest.mark.gpu


def _pack_both(w: torch.Tensor):
    mx = lib()
    wq, ws = mx.quantize(w)
    torch.cuda.synchronize()
    rq, rs = oracle.quantize(w.cpu().numpy())
    return wq, ws, rq, rs


def test_quantize_bitexact_adversarial_blocks():
    rng = np.random.default_rng(1)
    blocks = oracle_pins.random_blocks(rng, 4096)
    w = torch.from_numpy(blocks.reshape(128, 1024)).cuda()
    wq, ws, rq, rs = _pack_both(w)
    assert np.array_equal(ws.cpu().numpy(), rs)
    assert np.array_equal(wq.cpu().numpy(), rq)


@pytest.mark.parametrize("seed,n,k,x64", [(0, 1024, 1024, False), (1, 7168, 7168, False), (2, 640, 7168, True),
                                          (3, 33, 96, False), (4, 1, 32, False)])
def test_quantize_bitexact_workloads(seed, n, k, x64):
    w = synth.weights(seed, n, k, device="cuda", x64_blocks=x64)
    wq, ws, rq, rs = _pack_both(w)
    assert np.array_equal(ws.cpu().numpy(), rs)
    assert np.array_equal(wq.cpu().numpy(), rq)


@pytest.mark.parametrize("t,k,n", [(1, 1024, 1024), (4, 1024, 1024), (3, 96, 17), (5, 1056, 100), (8, 2080, 48),
                                   (2, 32, 1), (7, 512, 4096), (1, 8192, 260)])
def test_linear_small_shapes(t, k, n):
    mx = lib()
    w, x = linear_case(11 + t, t, k, n)
    wq, ws, rq, rs = _pack_both(w)
    yg = Guarded((t, n), torch.bfloat16)
    y = mx.linear(x, wq, ws, out=yg.t)
    yg.check(f"linear t={t} k={k} n={n}")
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"linear t={t} k={k} n={n}")


@pytest.mark.parametrize("t", [9, 16, 23, 32])
def test_linear_many_tokens(t):
    mx = lib()
    k, n = 2048, 300
    w, x = linear_case(40 + t, t, k, n)
    wq, ws, rq, rs = _pack_both(w)
    yg = Guarded((t, n), torch.bfloat16)
    y = mx.linear(x, wq, ws, out=yg.t)
    yg.check(f"linear t={t}")
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"linear t={t}")


@pytest.mark.parametrize("t,k,n", [(16, 7168, 130), (32, 7168, 70), (24, 14336, 40), (8, 16384, 33),
                                   (12, 30720, 17)])
def test_linear_cluster_split_k(t, k, n):
    """Token counts whose staged activations exceed one SM, with one row group
    per CTA: K is split over a thread-block cluster and the partial sums meet
    through DSMEM."""
    mx = lib()
    w, x = linear_case(60 + t, t, k, n)
    wq, ws, rq, rs = _pack_both(w)
    yg = Guarded((t, n), torch.bfloat16)
    y = mx.linear(x, wq, ws, out=yg.t)
    yg.check(f"cluster t={t} k={k} n={n}")
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"cluster t={t} k={k} n={n}")
    assert mx.last_device_status() == mx.MXFP4_OK


@pytest.mark.parametrize("t,k,n", [(16, 7168, 4900), (32, 7200, 4900), (12, 7168, 4864), (17, 4096, 5000),
                                   (24, 14336, 4900)])
def test_linear_k_parts(t, k, n):
    """Token counts whose activations over all of K leave no useful ring in
    one SM, with at least 2 row groups per CTA: each CTA walks K in parts
    (double-buffered activation parts; each row group's sums stay with one
    warp across the parts). Covers a ragged row group, K % 256 != 0 (29
    one-step parts, the last one block long), partial token tiles (12 of 16,
    17 of 32) and CTAs with fewer row groups than warps."""
    mx = lib()
    w, x = linear_case(80 + t, t, k, n)
    wq, ws, rq, rs = _pack_both(w)
    yg = Guarded((t, n), torch.bfloat16)
    y = mx.linear(x, wq, ws, out=yg.t)
    yg.check(f"k parts t={t} k={k} n={n}")
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"k parts t={t} k={k} n={n}")
    assert mx.last_device_status() == mx.MXFP4_OK


def test_linear_k_parts_many_batches_sampled():
    """T=32, K=4096, N=40008: 16-17 row groups per CTA in batches of 8 (one
    per consumer warp), so every CTA re-stages the activation parts per
    batch and a CTA with 17 ends on a one-unit batch; sampled rows
    (including the ragged last group of 8) against the oracle."""
    mx = lib()
    t, k, n = 32, 4096, 40008
    w, x = linear_case(90, t, k, n)
    wq, ws = mx.quantize(w)
    y = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    rows = np.union1d(sample_rows(n, 256, seed=90), np.arange(n - 16, n))
    rows_t = torch.from_numpy(rows).cuda()
    rq, rs = oracle.quantize(w[rows_t].cpu().numpy())
    del w
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y[:, rows_t]), y_ref, rss, "k parts, many batches")
    assert mx.last_device_status() == mx.MXFP4_OK


@pytest.mark.parametrize("t,k,n", [(5, 6144, 12000), (3, 6176, 10000)])
def test_linear_odd_stage_sizes_sampled(t, k, n):
    """More than 4 row groups per SM with activations that fit: whole-stage
    chunks of 8 / 5 steps. The second shape has K % 256 != 0 (25 steps, the
    last one block long), fetched through the 2D tensor map. Sampled rows,
    including the ragged tail."""
    mx = lib()
    plan = mx.linear_plan(t, k, n)
    assert plan["mode"] == 0 and plan["stage_steps"] == plan["chunk_steps"] >= 5, plan
    w, x = linear_case(100 + t, t, k, n)
    wq, ws = mx.quantize(w)
    y = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    rows = np.union1d(sample_rows(n, 384, seed=100 + t), np.arange(n - 20, n))
    rows_t = torch.from_numpy(rows).cuda()
    rq, rs = oracle.quantize(w[rows_t].cpu().numpy())
    del w
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y[:, rows_t]), y_ref, rss, f"odd stages t={t} k={k} n={n}")
    assert mx.last_device_status() == mx.MXFP4_OK


@pytest.mark.parametrize("t,k,n", [(1, 262144, 40), (32, 262144, 24)])
def test_linear_largest_k(t, k, n):
    """The largest k the header promises (262144): one row group's scales for
    all of k take 128 KB of shared memory, so each CTA walks K in parts
    (hundreds of them) with a single row group; ragged last row group."""
    mx = lib()
    assert mx.linear_plan(t, k, n)["mode"] == 1
    w, x = linear_case(110 + t, t, k, n)
    wq, ws, rq, rs = _pack_both(w)
    y = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"largest k t={t} n={n}")
    assert mx.last_device_status() == mx.MXFP4_OK


def test_linear_config1_full():
    """T=1, K=N=1024, seed 0: whole output against the oracle."""
    mx = lib()
    w, x = linear_case(0, 1, 1024, 1024)
    wq, ws, rq, rs = _pack_both(w)
    y = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, "config 1")


def test_linear_verify_t4_full():
    """T=4, K=N=7168 (one target + three drafts): whole output."""
    mx = lib()
    w, x = linear_case(1, 4, 7168, 7168)
    wq, ws, rq, rs = _pack_both(w)
    assert np.array_equal(wq.cpu().numpy(), rq) and np.array_equal(ws.cpu().numpy(), rs)
    y = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, "verify t=4")


def test_linear_lmhead_full_size_sampled():
    """LM head T=4, K=7168, N=129280 with 1% of blocks x64: packing of sampled
    rows bit-exact, sampled output rows within tolerance."""
    mx = lib()
    t, k, n = 4, 7168, 129280
    w, x = linear_case(2, t, k, n, x64=True)
    wq, ws = mx.quantize(w)
    y = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    rows = sample_rows(n, 384, seed=2)
    rows_t = torch.from_numpy(rows).cuda()
    rq, rs = oracle.quantize(w[rows_t].cpu().numpy())
    assert np.array_equal(wq[rows_t].cpu().numpy(), rq)
    assert np.array_equal(ws[rows_t].cpu().numpy(), rs)
    del w
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y[:, rows_t]), y_ref, rss, "lm head")


@pytest.mark.parametrize("t", [1, 2, 4, 8, 16, 32])
def test_linear_ffn_sweep_sampled(t):
    """K=7168, N=18432, one weight set (seed 3) reused across T."""
    mx = lib()
    k, n = 7168, 18432
    w = synth.weights(3, n, k, device="cuda")
    x = synth.tokens(3, t, k, device="cuda")
    wq, ws = mx.quantize(w)
    y = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    rows = sample_rows(n, 256, seed=t)
    rows_t = torch.from_numpy(rows).cuda()
    rq, rs = oracle.quantize(w[rows_t].cpu().numpy())
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y[:, rows_t]), y_ref, rss, f"ffn t={t}")


def test_linear_extreme_scales():
    """Blocks with scale bytes 0, 1, 2, 250, 252 and 254 next to ordinary ones;
    activations chosen so every exact output stays inside bf16 range."""
    mx = lib()
    rng = np.random.default_rng(5)
    t, k, n = 3, 512, 64
    rq = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    rs = rng.integers(120, 135, (n, k // 32), dtype=np.uint8)
    xs = rng.normal(0, 1, (t, k)).astype(np.float32)
    for r in range(n):
        kind = r % 6
        b = r % (k // 32)
        s = [0, 1, 2, 250, 252, 254][kind]
        rs[r, b] = s
        if s >= 250:  # shrink the matching activations so the product stays finite
            xs[:, b * 32:(b + 1) * 32] *= 2.0 ** -100
    x = torch.from_numpy(xs).to(torch.bfloat16)
    y = mx.linear(x.cuda(), torch.from_numpy(rq).cuda(), torch.from_numpy(rs).cuda())
    torch.cuda.synchronize()
    y_ref, rss = oracle.linear(x, rq, rs)
    assert np.all(np.abs(y_ref) < 3e38)
    assert_within(bf16_to_f64(y), y_ref, rss, "extreme scales")


def test_linear_activation_extremes():
    """bf16 activations spanning subnormal to 2^120, and all-zero blocks."""
    mx = lib()
    rng = np.random.default_rng(6)
    t, k, n = 4, 1024, 96
    xs = rng.normal(0, 1, (t, k)) * 2.0 ** rng.integers(-130, 100, (t, k // 32)).repeat(32, axis=1)
    xs[1, 64:96] = 0.0
    xs = np.clip(xs, -1e35, 1e35).astype(np.float32)
    x = torch.from_numpy(xs).to(torch.bfloat16)
    w = synth.weights(6, n, k) * 1e-3
    rq, rs = oracle.quantize(w.numpy())
    y = mx.linear(x.cuda(), torch.from_numpy(rq).cuda(), torch.from_numpy(rs).cuda())
    torch.cuda.synchronize()
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, "activation extremes")


def test_linear_deterministic():
    mx = lib()
    w, x = linear_case(8, 4, 7168, 2048)
    wq, ws = mx.quantize(w)
    y1 = mx.linear(x, wq, ws)
    y2 = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_linear_no_device_timeout():
    mx = lib()
    w, x = linear_case(9, 2, 1024, 512)
    wq, ws = mx.quantize(w)
    mx.linear(x, wq, ws)
    assert mx.last_device_status() == mx.MXFP4_OK
