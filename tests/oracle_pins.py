"""Pins for the CPU oracle: checks against things other than the oracle.

Each check takes an ``oracle.Oracle`` (so the mutation test can run the same
checks against copies of the oracle with planted mistakes) and raises
AssertionError on a mismatch. The references used here are independent of
the oracle's code: CUDA's host-side cuda_fp4.h / cuda_fp8.h conversions,
torch's float8_e8m0fnu dtype, exact rational arithmetic (fractions), numpy
matmul, scipy's softmax/expit, mpmath, Python's sort and closed forms that
follow from the format definition ("Zyphra Inference Wave 2", section
"Quantization": 32-value blocks, one power-of-two scale, magnitudes
0, 0.5, 1, 1.5, 2, 3, 4, 6).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---------------------------------------------------------------- helpers
def floor_log2_exact(a: float) -> int:
    """floor(log2 a) for a finite a > 0 from its exact rational value."""
    p, q = Fraction(a).as_integer_ratio()
    m = p.bit_length() - q.bit_length()
    # now 2^(m-1) < p/q < 2^(m+1); settle m exactly with integer compares
    while Fraction(p, q) < Fraction(2) ** m:
        m -= 1
    while Fraction(p, q) >= Fraction(2) ** (m + 1):
        m += 1
    return m


def expected_scale(block: np.ndarray) -> int:
    amax = float(np.max(np.abs(block.astype(np.float64))))
    if amax == 0.0:
        return 0
    return min(254, max(0, floor_log2_exact(amax) - 2 + 127))


def lib_decode(pin, wq: np.ndarray, ws: np.ndarray) -> np.ndarray:
    """Dequantize with the library routines only (cuda_fp4 codes, torch E8M0)."""
    codes = np.stack([wq & 15, wq >> 4], axis=-1).reshape(wq.shape[0], -1)
    table = np.array([pin.pin_e2m1_decode(c) for c in range(16)], np.float64)
    scale = torch.from_numpy(ws.copy()).view(torch.float8_e8m0fnu).float().double().numpy()
    return table[codes] * np.repeat(scale, 32, axis=1)


def bf16_round(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def random_blocks(rng: np.random.Generator, nblocks: int) -> np.ndarray:
    """Blocks of 32 float32 with varied magnitudes, ties, zeros and signed zeros."""
    out = []
    for i in range(nblocks):
        kind = i % 6
        if kind == 0:
            b = rng.normal(0, 0.02, 32)
        elif kind == 1:
            b = rng.normal(0, 1, 32) * 64.0
        elif kind == 2:  # exact grid multiples of a power of two, including ties
            b = rng.choice([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6], 32)
            b = b * rng.choice([-1, 1], 32) * 2.0 ** rng.integers(-10, 10)
        elif kind == 3:  # fp32 subnormals and tiny normals
            b = rng.normal(0, 1, 32) * 2.0 ** rng.integers(-149, -120)
        elif kind == 4:  # values that round to zero keep their sign
            b = rng.normal(0, 1e-3, 32)
            b[0] = 1.0
            b[1] = -0.0
        else:
            b = np.zeros(32)
            b[rng.integers(0, 32)] = -0.0
        out.append(np.asarray(b, np.float32))
    return np.stack(out)


# ----------------------------------------------------------- format pins
def check_decode_table(orc, pin):
    for c in range(16):
        got, ref = orc.e2m1_value(c), float(pin.pin_e2m1_decode(c))
        assert got == ref and math.copysign(1, got) == math.copysign(1, ref), (c, got, ref)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).float().double().numpy()
    for s in range(255):
        assert orc.e8m0_value(s) == ref[s], (s, orc.e8m0_value(s), ref[s])
        assert orc.e8m0_value(s) == float(pin.pin_e8m0_decode(s))
    assert math.isnan(orc.e8m0_value(255)) and math.isnan(ref[255])


def rounding_points():
    pts = [i / 64 for i in range(0, 8 * 64 + 1)]
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for t in ties:
        pts += [t, math.nextafter(t, 0), math.nextafter(t, 10), t - 2 ** -30, t + 2 ** -30]
    pts += [6.0, 6.5, 7.0, 7.999, 100.0, 1e30, 2 ** -20, 0.0]
    return pts


def check_rounding(orc, pin):
    for a in rounding_points():
        assert orc.e2m1_round_magnitude(a) == pin.pin_e2m1_round(a) & 7, (a, orc.e2m1_round_magnitude(a))
    # the stated tie table: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    for a, v in [(0.25, 0), (0.75, 1), (1.25, 1), (1.75, 2), (2.5, 2), (3.5, 4), (5.0, 4), (6.5, 6), (7.5, 6)]:
        assert E2M1_GRID[orc.e2m1_round_magnitude(a)] == v, a


def check_block_scale(orc):
    rng = np.random.default_rng(7)
    amaxes = []
    for k in range(-149, 128):
        p = 2.0 ** k
        amaxes += [p, float(np.nextafter(np.float32(p), np.float32(0))), float(np.nextafter(np.float32(p), np.float32(np.inf)))]
    amaxes += list(rng.uniform(0, 1, 50)) + list(rng.normal(0, 0.02, 50)) + [0.0, 3.4e38]
    for a in amaxes:
        a32 = np.float32(a)
        if not np.isfinite(a32):
            continue
        b = (rng.uniform(-1, 1, 32) * a32).astype(np.float32)
        b[rng.integers(0, 32)] = -a32 if rng.integers(0, 2) else a32
        assert orc.block_scale(b) == expected_scale(b), (a, orc.block_scale(b), expected_scale(b))


def check_quantize(orc, pin):
    rng = np.random.default_rng(11)
    blocks = random_blocks(rng, 120)
    w = blocks.reshape(30, 128)
    wq, ws = orc.quantize(w)
    assert wq.shape == (30, 64) and ws.shape == (30, 4)
    for r in range(30):
        for b in range(4):
            blk = w[r, b * 32:(b + 1) * 32]
            s = expected_scale(blk)
            assert ws[r, b] == s, (r, b, ws[r, b], s)
            for i in range(32):
                v = float(blk[i]) * 2.0 ** (127 - s)  # exact: power-of-two scaling in float64
                code = pin.pin_e2m1_round(v)
                if math.copysign(1.0, float(blk[i])) < 0:
                    code |= 8  # the sign bit is kept even when the value rounds to zero
                byte = int(wq[r, b * 16 + i // 2])
                got = (byte >> 4) if i % 2 else (byte & 15)
                assert got == code, (r, b, i, float(blk[i]), got, code)


def check_all_ones(orc):
    wq, ws = orc.quantize(np.ones((4, 96), np.float32))
    # amax = 1 -> floor(log2 1) - 2 = -2 -> s = 125; 1 / 2^-2 = 4 = code 6
    assert (wq == 0x66).all() and (ws == 125).all()
    assert (orc.dequant(wq, ws) == 1.0).all()


def check_round_trip(orc):
    rng = np.random.default_rng(3)
    n = 64
    codes = rng.integers(0, 16, (n, 64))
    codes[:, 0] = rng.choice([6, 7, 14, 15], n)  # block max magnitude 4 or 6 in each block
    codes[:, 32] = rng.choice([6, 7, 14, 15], n)
    s = rng.integers(2, 250, (n, 2))
    vals = np.array([E2M1_GRID[c & 7] * (-1 if c & 8 else 1) for c in codes.ravel()]).reshape(n, 64)
    w = (vals * np.repeat(2.0 ** (s - 127.0), 32, axis=1)).astype(np.float32)
    wq, ws = orc.quantize(w)
    want = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    # -0.0 is encoded as code 8, and the float input for code 8 is -0.0: identical
    assert (ws == s).all()
    assert (wq == want).all()
    # value idempotence for any block: dequant(quantize(dequant(q))) == dequant(q)
    codes2 = rng.integers(0, 16, (n, 64))
    s2 = rng.integers(20, 230, (n, 2))
    q2 = (codes2[:, 0::2] | (codes2[:, 1::2] << 4)).astype(np.uint8)
    d = orc.dequant(q2, s2.astype(np.uint8))
    wq3, ws3 = orc.quantize(d.astype(np.float32))
    assert (orc.dequant(wq3, ws3) == d).all()


def check_dequant(orc, pin):
    rng = np.random.default_rng(5)
    wq = rng.integers(0, 256, (16, 48), dtype=np.uint8)
    ws = rng.integers(0, 255, (16, 3), dtype=np.uint8)
    assert np.array_equal(orc.dequant(wq, ws), lib_decode(pin, wq, ws))


# ----------------------------------------------------------- linear pins
def check_linear_all_ones_codes(orc):
    rng = np.random.default_rng(9)
    t, k, n = 3, 1024, 5
    x = bf16_round(rng.normal(0, 1, (t, k)))
    wq = np.full((n, k // 2), 0x22, np.uint8)  # two codes of value 1.0 per byte
    ws = np.full((n, k // 32), 127, np.uint8)  # scale 2^0
    y, _ = orc.linear(x, wq, ws)
    xs = x.float().double().numpy()
    for ti in range(t):
        ref = math.fsum(xs[ti])
        assert np.all(np.abs(y[ti] - ref) <= 2.0 ** -50 * np.abs(xs[ti]).sum()), (y[ti], ref)


def check_linear_fraction(orc, pin):
    rng = np.random.default_rng(13)
    table = [Fraction(pin.pin_e2m1_decode(c)) for c in range(16)]
    for t, k, n in [(1, 32, 3), (3, 64, 5), (2, 96, 8)]:
        x = bf16_round(rng.normal(0, 1, (t, k)))
        wq = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
        ws = rng.integers(118, 136, (n, k // 32), dtype=np.uint8)
        y, rss = orc.linear(x, wq, ws)
        xs = x.float().double().numpy()
        for ti in range(t):
            for r in range(n):
                acc = Fraction(0)
                sq = Fraction(0)
                mag = 0.0
                for c in range(k):
                    byte = int(wq[r, c // 2])
                    code = (byte >> 4) if c % 2 else (byte & 15)
                    wv = table[code] * Fraction(2) ** (int(ws[r, c // 32]) - 127)
                    p = Fraction(float(xs[ti, c])) * wv
                    acc += p
                    sq += p * p
                    mag += abs(float(p))
                assert abs(y[ti, r] - float(acc)) <= 1e-14 * mag + 1e-300, (t, k, n, ti, r)
                assert abs(rss[ti, r] - math.sqrt(float(sq))) <= 1e-14 * math.sqrt(float(sq)) + 1e-300


def check_linear_matmul(orc, pin):
    rng = np.random.default_rng(17)
    t, k, n = 4, 256, 40
    x = bf16_round(rng.normal(0, 1, (t, k)))
    wq = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    ws = rng.integers(110, 140, (n, k // 32), dtype=np.uint8)
    wd = lib_decode(pin, wq, ws)
    xs = x.float().double().numpy()
    ref = xs @ wd.T
    mag = np.abs(xs) @ np.abs(wd).T
    y, rss = orc.linear(x, wq, ws)
    assert np.all(np.abs(y - ref) <= 1e-13 * mag)
    assert np.allclose(rss, np.sqrt((xs ** 2) @ (wd ** 2).T), rtol=1e-12, atol=0)
    # a row subset returns the same values
    rows = np.array([3, 0, 39, 7])
    y2, _ = orc.linear(x, wq, ws, rows)
    assert np.array_equal(y2, y[:, rows])
    # one-hot rows: row r holds a single 1.0 at column c_r -> y = x[:, c_r]
    cols = rng.integers(0, k, n)
    wq1 = np.zeros((n, k // 2), np.uint8)
    for r, c in enumerate(cols):
        wq1[r, c // 2] = 0x02 << (4 * (c % 2))
    ws1 = np.full((n, k // 32), 127, np.uint8)
    y1, _ = orc.linear(x, wq1, ws1)
    assert np.array_equal(y1, xs[:, cols])


# -------------------------------------------------------------- MoE pins
def check_route(orc):
    from scipy.special import softmax
    rng = np.random.default_rng(19)
    lg = rng.normal(0, 1, (16, 64)).astype(np.float32)
    lg[3, 10] = lg[3, 20] = lg[3, 30] = 5.0  # ties resolve to the smaller index
    ids, g = orc.route(lg, 8)
    for ti in range(16):
        want = sorted(range(64), key=lambda c: (-float(lg[ti, c]), c))[:8]
        assert list(ids[ti]) == want, (ti, ids[ti], want)
        assert np.allclose(g[ti], softmax(lg[ti, want].astype(np.float64)), rtol=1e-14, atol=0)
        assert abs(g[ti].sum() - 1.0) <= 1e-15
    ids, g = orc.route(np.zeros((2, 256), np.float32), 8)
    assert (ids == np.arange(8)).all() and (g == 0.125).all()


def _pack(rng, n, k, smin=120, smax=132):
    wq = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    ws = rng.integers(smin, smax, (n, k // 32), dtype=np.uint8)
    return wq, ws


def check_moe_top1(orc, pin):
    from scipy.special import expit
    rng = np.random.default_rng(23)
    e, hidden, inter, t = 6, 64, 96, 5
    w1 = {ex: _pack(rng, 2 * inter, hidden) for ex in range(e)}
    w2 = {ex: _pack(rng, hidden, inter) for ex in range(e)}
    x = bf16_round(rng.normal(0, 1, (t, hidden)))
    lg = rng.normal(0, 1, (t, e)).astype(np.float32)
    y, _ = orc.moe(x, lg, 1, w1, w2, inter)
    xs = x.float().double().numpy()
    for ti in range(t):
        ex = int(np.argmax(lg[ti]))
        W1 = lib_decode(pin, *w1[ex])
        W2 = lib_decode(pin, *w2[ex])
        a = W1[:inter] @ xs[ti]
        b = W1[inter:] @ xs[ti]
        h = a * expit(a) * b  # SiLU(a) = a * sigmoid(a)
        ref = W2 @ h
        assert np.allclose(y[ti], ref, rtol=1e-10, atol=1e-12 * np.abs(W2) @ np.abs(h)), ti


def check_moe_shared(orc, pin):
    """Two shared experts after the routed top-2: each adds its own SwiGLU
    FFN output with weight 1 ("Zyphra Inference Wave 2", section
    "Quantization": a token uses its top-k routed experts plus the layer's
    shared experts)."""
    from scipy.special import expit, softmax
    rng = np.random.default_rng(31)
    e, ns, hidden, inter, t, top_k = 5, 2, 64, 32, 4, 2
    w1 = {ex: _pack(rng, 2 * inter, hidden) for ex in range(e + ns)}
    w2 = {ex: _pack(rng, hidden, inter) for ex in range(e + ns)}
    x = bf16_round(rng.normal(0, 1, (t, hidden)))
    lg = rng.normal(0, 1, (t, e)).astype(np.float32)
    y, _ = orc.moe(x, lg, top_k, w1, w2, inter, n_shared=ns)
    xs = x.float().double().numpy()

    def ffn(ex, xt):
        W1 = lib_decode(pin, *w1[ex])
        a, b = W1[:inter] @ xt, W1[inter:] @ xt
        return lib_decode(pin, *w2[ex]) @ (a * expit(a) * b)

    for ti in range(t):
        order = sorted(range(e), key=lambda c: (-float(lg[ti, c]), c))[:top_k]
        g = softmax(lg[ti, order].astype(np.float64))
        ref = sum(gi * ffn(ex, xs[ti]) for gi, ex in zip(g, order)) + sum(ffn(e + s, xs[ti]) for s in range(ns))
        mag = sum(np.abs(ffn(ex, xs[ti])) for ex in range(e + ns))
        assert np.allclose(y[ti], ref, rtol=1e-10, atol=1e-12 * float(mag.max())), ti
    # With no shared expert the call is the routed MoE itself.
    y0, _ = orc.moe(x, lg, top_k, w1, w2, inter)
    y0s, _ = orc.moe(x, lg, top_k, w1, w2, inter, n_shared=0)
    assert np.array_equal(y0, y0s)


def check_moe_mpmath(orc, pin):
    import mpmath
    mpmath.mp.dps = 40
    rng = np.random.default_rng(29)
    e, hidden, inter, t, top_k = 5, 32, 64, 3, 3
    w1 = {ex: _pack(rng, 2 * inter, hidden) for ex in range(e)}
    w2 = {ex: _pack(rng, hidden, inter) for ex in range(e)}
    x = bf16_round(rng.normal(0, 1, (t, hidden)))
    lg = rng.normal(0, 1, (t, e)).astype(np.float32)
    y, rss = orc.moe(x, lg, top_k, w1, w2, inter)
    xs = x.float().double().numpy()
    dec1 = {ex: lib_decode(pin, *w1[ex]) for ex in range(e)}
    dec2 = {ex: lib_decode(pin, *w2[ex]) for ex in range(e)}
    for ti in range(t):
        order = sorted(range(e), key=lambda c: (-float(lg[ti, c]), c))[:top_k]
        ex_l = [mpmath.exp(mpmath.mpf(float(lg[ti, c]))) for c in order]
        z = sum(ex_l)
        gs = [v / z for v in ex_l]
        out = [mpmath.mpf(0)] * hidden
        sq = [mpmath.mpf(0)] * hidden
        for gi, ex in zip(gs, order):
            h = []
            for r in range(inter):
                a = mpmath.fsum(mpmath.mpf(float(xs[ti, c])) * mpmath.mpf(float(dec1[ex][r, c])) for c in range(hidden))
                b = mpmath.fsum(mpmath.mpf(float(xs[ti, c])) * mpmath.mpf(float(dec1[ex][r + inter, c])) for c in range(hidden))
                h.append(a / (1 + mpmath.exp(-a)) * b)
            for n in range(hidden):
                terms = [h[j] * mpmath.mpf(float(dec2[ex][n, j])) for j in range(inter)]
                out[n] += gi * mpmath.fsum(terms)
                sq[n] += mpmath.fsum((gi * tt) ** 2 for tt in terms)
        for n in range(hidden):
            ref = float(out[n])
            assert abs(y[ti, n] - ref) <= 1e-12 * float(mpmath.sqrt(sq[n])) * inter, (ti, n, y[ti, n], ref)
            assert abs(rss[ti, n] - float(mpmath.sqrt(sq[n]))) <= 1e-12 * float(mpmath.sqrt(sq[n]))


ALL_CHECKS = [
    ("decode_table", check_decode_table, True),
    ("rounding", check_rounding, True),
    ("block_scale", check_block_scale, False),
    ("quantize", check_quantize, True),
    ("all_ones", check_all_ones, False),
    ("round_trip", check_round_trip, False),
    ("dequant", check_dequant, True),
    ("linear_all_ones_codes", check_linear_all_ones_codes, False),
    ("linear_fraction", check_linear_fraction, True),
    ("linear_matmul", check_linear_matmul, True),
    ("route", check_route, False),
    ("moe_top1", check_moe_top1, True),
    ("moe_mpmath", check_moe_mpmath, True),
    ("moe_shared", check_moe_shared, True),
]


def run_all(orc, pin):
    """Run every check; returns the list of names that failed."""
    failed = []
    for name, fn, needs_pin in ALL_CHECKS:
        try:
            fn(orc, pin) if needs_pin else fn(orc)
        except AssertionError:
            failed.append(name)
    return failed
