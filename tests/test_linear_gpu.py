"""GPU parity of mxfp4_quantize and mxfp4_linear against the oracle.

Packing is compared byte for byte; outputs elementwise under the stated
bound |y - y_ref| <= 4e-3*|y_ref| + 1e-3*sqrt(sum_k (x_k*w_k)^2).

mxfp4_linear has three kernels: the packed-E2M1 tensor-core kernel for
t <= 8 and k % 512 == 0 (plan mode 4), the E4M3-split tensor-core kernel
for t >= 9 and k % 512 == 0 (mode 3) and the streaming engine otherwise
(modes 0-2). Shapes below cover all three; k % 512 != 0 twins keep the
engine's whole-K, K-in-parts and cluster modes under test.
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


@pytest.mark.parametrize("t,k", [(9, 2048), (16, 2048), (23, 2048), (32, 2048), (9, 2080), (32, 2080)])
def test_linear_many_tokens(t, k):
    mx = lib()
    n = 300
    w, x = linear_case(40 + t, t, k, n)
    wq, ws, rq, rs = _pack_both(w)
    yg = Guarded((t, n), torch.bfloat16)
    y = mx.linear(x, wq, ws, out=yg.t)
    yg.check(f"linear t={t}")
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"linear t={t}")


@pytest.mark.parametrize("t,k,n", [(16, 7168, 130), (32, 7168, 70), (24, 14336, 40), (8, 16384, 33),
                                   (12, 30720, 17), (16, 7200, 130), (8, 16416, 33)])
def test_linear_cluster_split_k(t, k, n):
    """Few output rows for many tokens and a long K: K is split over the two
    CTAs of a cluster and the partial sums meet through distributed shared
    memory (tensor-core kernel for k % 512 == 0; the engine's cluster mode
    for the last two shapes)."""
    mx = lib()
    plan = mx.linear_plan(t, k, n)
    assert plan["cluster"] == 2 or plan["mode"] == 1, plan
    mx = lib()
    w, x = linear_case(60 + t, t, k, n)
    wq, ws, rq, rs = _pack_both(w)
    yg = Guarded((t, n), torch.bfloat16)
    y = mx.linear(x, wq, ws, out=yg.t)
    yg.check(f"cluster t={t} k={k} n={n}")
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"cluster t={t} k={k} n={n}")
    assert mx.last_device_status() == mx.MXFP4_OK


@pytest.mark.parametrize("t,k,n", [(16, 7200, 4900), (32, 7200, 4900), (12, 7200, 4864), (17, 4128, 5000),
                                   (24, 14368, 4900), (16, 7168, 4900), (17, 4096, 5000)])
def test_linear_k_parts(t, k, n):
    """Streaming engine (k % 512 != 0), token counts whose activations over
    all of K leave no useful ring in one SM, with at least 2 row groups per
    CTA: each CTA walks K in parts (double-buffered activation parts; each
    row group's sums stay with one warp across the parts). Covers a ragged
    row group, K % 256 != 0 (29 one-step parts, the last one block long),
    partial token tiles (12 of 16, 17 of 32) and CTAs with fewer row groups
    than warps. The last two shapes are the same sizes on the tensor-core
    kernels (t = 16: packed E2M1, 69 clusters of 72 rows; t = 17: E4M3 split,
    2-CTA clusters over 39-40 tiles of 128 rows, ragged last tile)."""
    mx = lib()
    assert mx.linear_plan(t, k, n)["mode"] == (1 if k % 512 else (4 if t <= 16 else 3))
    w, x = linear_case(80 + t, t, k, n)
    wq, ws, rq, rs = _pack_both(w)
    yg = Guarded((t, n), torch.bfloat16)
    y = mx.linear(x, wq, ws, out=yg.t)
    yg.check(f"k parts t={t} k={k} n={n}")
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"k parts t={t} k={k} n={n}")
    assert mx.last_device_status() == mx.MXFP4_OK


@pytest.mark.parametrize("k", [4128, 4096])
def test_linear_k_parts_many_batches_sampled(k):
    """T=32, N=40008. K=4128 (streaming engine): 16-17 row groups per CTA in
    batches of 8 (one per consumer warp), so every CTA re-stages the
    activation parts per batch and a CTA with 17 ends on a one-unit batch.
    K=4096 (tensor-core kernel): 313 tiles of 128 rows, 2-3 per CTA, the
    last one 72 rows. Sampled rows (including the ragged tail) against the
    oracle."""
    mx = lib()
    t, n = 32, 40008
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


@pytest.mark.parametrize("t,k,n", [(5, 6112, 12000), (3, 6176, 10000)])
def test_linear_odd_stage_sizes_sampled(t, k, n):
    """Streaming engine, more than 4 row groups per SM with activations that
    fit: whole-stage chunks of 8 / 5 steps. Both shapes have K % 256 != 0
    (24 and 25 steps, the last one a partial step), fetched through the 2D
    tensor map. Sampled rows, including the ragged tail."""
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


@pytest.mark.parametrize("t,k,n", [(1, 262144, 40), (32, 262144, 24), (1, 262112, 40), (32, 262112, 24)])
def test_linear_largest_k(t, k, n):
    """The largest k the header promises (262144). Tensor-core kernels: one
    tile per 2-CTA cluster, 256 stages per CTA (t = 1: packed E2M1, groups
    of 8 rows; t = 32: E4M3 split). Streaming engine
    (k = 262112): one row group's scales for all of k take 128 KB of shared
    memory, so each CTA walks K in parts (hundreds of them) with a single
    row group; ragged last row group."""
    mx = lib()
    assert mx.linear_plan(t, k, n)["mode"] == ((4 if t <= 16 else 3) if k % 512 == 0 else 1)
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


@pytest.mark.parametrize("t", [4, 8])
def test_linear_verify_full(t):
    """K=N=7168, whole output: T=4 (one target + three drafts) and T=8, both
    on the packed-E2M1 kernel (75 clusters of 2 CTAs, 96 rows each)."""
    mx = lib()
    w, x = linear_case(1, t, 7168, 7168)
    wq, ws, rq, rs = _pack_both(w)
    assert np.array_equal(wq.cpu().numpy(), rq) and np.array_equal(ws.cpu().numpy(), rs)
    y = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y), y_ref, rss, f"verify t={t}")


@pytest.mark.parametrize("t", [4, 6])
def test_linear_lmhead_full_size_sampled(t):
    """LM head K=7168, N=129280 with 1% of blocks x64 (T=4 as configured,
    and T=6): the packed-E2M1 kernel, 856 rows per CTA in six 128-row tiles
    and one of 88 rows, one batch; the last CTA holds 24 rows):
    packing of sampled rows bit-exact, sampled output rows within tolerance."""
    mx = lib()
    k, n = 7168, 129280
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


@pytest.mark.parametrize("t", [1, 2, 4, 5, 7, 8, 12, 16, 32])
def test_linear_ffn_sweep_sampled(t):
    """K=7168, N=18432, one weight set (seed 3) reused across T (t = 5-16:
    2-CTA clusters over 248 rows; t = 32: the E4M3-split kernel)."""
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


@pytest.mark.parametrize("t,k", [(5, 512), (3, 512), (3, 544)])
def test_linear_extreme_scales(t, k):
    """Blocks with scale bytes 0, 1, 2, 250, 252 and 254 next to ordinary ones;
    activations chosen so every exact output stays inside bf16 range (t = 5
    and t = 3 at k = 512: packed-E2M1 kernel; k = 544: streaming engine)."""
    mx = lib()
    rng = np.random.default_rng(5)
    n = 64
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


@pytest.mark.parametrize("t,k", [(4, 1024), (6, 1024), (6, 1056)])
def test_linear_activation_extremes(t, k):
    """bf16 activations spanning subnormal to 2^120, and all-zero blocks
    (k = 1024: packed-E2M1 kernel; k = 1056: streaming engine)."""
    mx = lib()
    rng = np.random.default_rng(6)
    n = 96
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


@pytest.mark.parametrize("t", [4, 8])
def test_linear_deterministic(t):
    mx = lib()
    w, x = linear_case(8, t, 7168, 2048)
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


@pytest.mark.parametrize("t,k", [(6, 512), (2, 512), (2, 544)])
def test_linear_scale_times_activation_factor_no_overflow(t, k):
    """Blocks with weight scale 2^127 (s = 254) whose nonzero codes meet
    small activations, while a larger activation of the same 32-block meets
    a zero code. The exact result is finite, but the weight scale times the
    activation block's own power-of-two factor reaches 2^128: no kernel may
    form that product on its way to the result. The large activation is 2^8
    (E4M3-split kernel: its activation scale is 2^1) and 2^16 (streaming
    engine, k = 544: its staging factor is 2^2); the small ones
    are +-2^-5 times a 4-bit significand, so every piece of them stays
    exact, and the weight codes of the block are +-0.5, which keeps every
    exact output below 2^127. On the packed-E2M1 kernel (k = 512) the large
    activation is 2^2: its digit pieces hold values down to 2^-13 exactly,
    and the weight scale times the top piece's scale is 2^129."""
    mx = lib()
    rng = np.random.default_rng(12)
    n = 48
    big = {3: 2.0 ** 8, 4: 2.0 ** 2}.get(mx.linear_plan(t, k, n)["mode"], 2.0 ** 16)
    rq = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    rs = rng.integers(120, 126, (n, k // 32), dtype=np.uint8)
    xs = rng.normal(0, 1, (t, k)).astype(np.float32)
    b0 = 3  # the extreme block
    xs[:, b0 * 32:(b0 + 1) * 32] = (2.0 ** -5) * (1 + rng.integers(0, 8, (t, 32)) / 8.0) * \
        rng.choice([-1.0, 1.0], (t, 32))
    xs[:, b0 * 32 + 5] = big
    codes = np.zeros((n, 32), np.uint8)
    codes[:, :] = rng.choice([1, 9], (n, 32))  # +-0.5
    codes[:, 5] = 0                                   # the large activation meets a zero weight
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    rq[:, b0 * 16:(b0 + 1) * 16] = packed
    rs[:, b0] = 254
    x = torch.from_numpy(xs).to(torch.bfloat16)
    blk = slice(b0 * 32, (b0 + 1) * 32)
    assert np.array_equal(x.float().numpy()[:, blk], xs[:, blk])  # the constructed block is exact in bf16
    y = mx.linear(x.cuda(), torch.from_numpy(rq).cuda(), torch.from_numpy(rs).cuda())
    torch.cuda.synchronize()
    y_ref, rss = oracle.linear(x, rq, rs)
    assert np.all(np.isfinite(y_ref)) and np.all(np.abs(y_ref) < 2.0 ** 127)
    yg = bf16_to_f64(y)
    assert np.all(np.isfinite(yg)), "overflow"
    assert_within(yg, y_ref, rss, f"scale x factor, k={k}")


@pytest.mark.parametrize("t,k", [(1, 1024), (4, 2048), (8, 1024)])
def test_linear_digit_pieces_exact(t, k):
    """Packed-E2M1 kernel: one weight of 1.0 per row (code 2, scale 2^0)
    makes y[t][n] = x[t][k_n], so y shows each activation as the kernel's
    digit pieces rebuild it. Within 2^8 of its block's largest magnitude a
    bf16 activation is rebuilt exactly, so y equals x bit for bit; further
    below, the error is at most 2^(E-16) (E = floor(log2) of the block
    maximum), and the oracle's tolerance holds for every output."""
    mx = lib()
    n = 2 * k // 32
    assert mx.linear_plan(t, k, n)["mode"] == 4
    rng = np.random.default_rng(13)
    # Activations: per 32-block one magnitude 2^e0 and elements spread over
    # 2^e0 .. 2^(e0 - 12); one all-zero block. (Block maxima stay above
    # 2^-112: the lowest piece scale is 2^-127, so smaller blocks lose their
    # values below 2^-128.)
    e0 = rng.integers(-100, 100, (t, k // 32)).repeat(32, axis=1)
    xs = rng.choice([-1.0, 1.0], (t, k)) * (1 + rng.random((t, k))) * 2.0 ** (e0 - rng.integers(0, 13, (t, k)))
    xs[:, 0:32] = 0.0
    x = torch.from_numpy(xs.astype(np.float32)).to(torch.bfloat16)
    xf = x.double().numpy()
    # Row r selects k_r: two rows per block (a large and a small element).
    kr = np.empty(n, np.int64)
    for b in range(k // 32):
        mags = np.abs(xf[0, 32 * b:32 * b + 32])
        kr[2 * b] = 32 * b + int(np.argmax(mags))
        kr[2 * b + 1] = 32 * b + int(np.argmin(np.where(mags > 0, mags, np.inf))) if (mags > 0).any() else 32 * b
    codes = np.zeros((n, k), np.uint8)
    codes[np.arange(n), kr] = 2  # 1.0
    rq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    rs = np.full((n, k // 32), 127, np.uint8)
    y = mx.linear(x.cuda(), torch.from_numpy(rq).cuda(), torch.from_numpy(rs).cuda())
    torch.cuda.synchronize()
    yg = bf16_to_f64(y)
    y_ref, rss = oracle.linear(x, rq, rs)
    sel = xf[:, kr]  # [t, n]: the selected activation of each output
    assert np.array_equal(y_ref, sel)
    blk_max = np.abs(xf).reshape(t, k // 32, 32).max(axis=2)[:, kr // 32]
    near = (np.abs(sel) * 2.0 ** 8 >= blk_max) | (sel == 0)
    assert near.any() and (~near).any()
    assert np.array_equal(yg[near], sel[near]), "values within 2^8 of the block maximum are exact"
    # (A one-hot row's tolerance is 5e-3 of the value itself, tighter than
    # the split's bound for elements far below their block maximum; those
    # are checked against the bound below instead.)
    assert_within(yg[near], y_ref[near], rss[near], "digit pieces")
    e_blk = np.floor(np.log2(np.where(blk_max > 0, blk_max, 1.0)))
    bound = 2.0 ** (np.maximum(e_blk, -112) - 16)
    # y is the rebuilt value rounded to bf16: at most the piece error plus half a bf16 ulp of it.
    err = np.abs(yg - sel)
    assert np.all(err[~near] <= bound[~near] + np.abs(sel[~near]) * 2.0 ** -8)
