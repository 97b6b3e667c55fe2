"""Seeded synthetic inputs for the MXFP4 weight-streaming workloads.

This module is shared by the CPU oracle tests, the GPU parity tests and the
bench. It draws random numbers and nothing else: it holds none of the MXFP4
arithmetic (no scale rule, no rounding, no packing, no dot products).

Generator (device independent, counter based):
  * 32-bit hash: the "lowbias32" integer mixer from Chris Wellons' hash
    prospector (xor-shift 16, multiply 0x7feb352d, xor-shift 15, multiply
    0x846ca68b, xor-shift 16, all modulo 2^32).
  * Each value is addressed by (seed, tensor id, stream, flat index). The
    flat index is split into its low and high 32-bit halves and each half is
    mixed with a key derived from (seed, tensor id, stream).
  * Normals: Box-Muller on two such uniforms, evaluated in float64 and
    rounded once to float32.
All integer work is exact in int64 (products are split so they never exceed
2^63), so CPU and CUDA produce identical uniforms; the float64 transform may
differ in the last ulp between devices, which parity never relies on: every
test generates a tensor once and hands the same bytes to both sides.

Workload recipes (shapes from the pages' decode-step configurations):
  * weights  W ~ N(0, 0.02) float32 (0.02 is the standard deviation)
  * tokens   x ~ N(0, 1) float32, rounded to bfloat16 (round to nearest even)
  * router logits ~ N(0, 1) float32
  * LM head: each 32-element K-block is independently selected with
    probability 0.01 and multiplied by 64 (exact in float32)
Tensor ids: W or W1 = 0, x = 1, logits = 2, W2 = 3, x64 block mask = 4.
"""
from __future__ import annotations

import math

import torch

MASK32 = 0xFFFFFFFF
TID_W = 0
TID_X = 1
TID_LOGITS = 2
TID_W2 = 3
TID_MASK = 4
MASK_THRESHOLD = 42949673  # round(0.01 * 2^32): P(u32 < threshold) = 0.01

_CHUNK = 1 << 24


def _mulmod32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for int64 x in [0, 2^32) without int64 overflow."""
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & MASK32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mulmod32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mulmod32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _mix32_int(v: int) -> int:
    t = torch.tensor([v & MASK32], dtype=torch.int64)
    return int(_mix32(t)[0])


def _keys(seed: int, tid: int, stream: int) -> tuple[int, int]:
    base = _mix32_int(seed) ^ _mix32_int(0x9E3779B9 * (tid + 1))
    k1 = _mix32_int(base ^ (0x85EBCA6B * (2 * stream + 1)))
    k2 = _mix32_int(k1 ^ 0xC2B2AE35)
    return k1, k2


def uint32_at(seed: int, tid: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """32-bit hash values (as int64) for flat indices ``idx`` (int64, >= 0)."""
    k1, k2 = _keys(seed, tid, stream)
    lo = idx & MASK32
    hi = idx >> 32
    return _mix32(_mix32(lo ^ k1) ^ _mix32(hi ^ k2))


def _normal_at(seed: int, tid: int, idx: torch.Tensor) -> torch.Tensor:
    a = uint32_at(seed, tid, 0, idx).to(torch.float64)
    b = uint32_at(seed, tid, 1, idx).to(torch.float64)
    u1 = (a + 0.5) * (1.0 / 4294967296.0)
    u2 = b * (1.0 / 4294967296.0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal(seed: int, tid: int, shape, sigma: float = 1.0, device="cpu",
           offset: int = 0) -> torch.Tensor:
    """float32 tensor of N(0, sigma^2) values, element i drawn at flat index offset+i."""
    numel = 1
    for s in shape:
        numel *= int(s)
    out = torch.empty(numel, dtype=torch.float32, device=device)
    for start in range(0, numel, _CHUNK):
        stop = min(numel, start + _CHUNK)
        idx = torch.arange(offset + start, offset + stop, dtype=torch.int64, device=device)
        out[start:stop] = (_normal_at(seed, tid, idx) * sigma).to(torch.float32)
    return out.view(*shape)


def weights(seed: int, n: int, k: int, tid: int = TID_W, sigma: float = 0.02,
            device="cpu", row0: int = 0, x64_blocks: bool = False) -> torch.Tensor:
    """W[n, k] float32 ~ N(0, sigma); rows row0..row0+n-1 of a larger matrix.

    With ``x64_blocks`` each 32-element K-block is selected with probability
    0.01 (hash of tensor id 4 at the block's flat index) and scaled by 64.
    """
    w = normal(seed, tid, (n, k), sigma, device, offset=row0 * k)
    if x64_blocks:
        w *= block_x64_mask(seed, n, k, device, row0).repeat_interleave(32, dim=1).to(w.dtype) * 63.0 + 1.0
    return w


def block_x64_mask(seed: int, n: int, k: int, device="cpu", row0: int = 0) -> torch.Tensor:
    """bool[n, k/32]: which 32-blocks of rows row0..row0+n-1 are scaled by 64."""
    nb = k // 32
    out = torch.empty(n * nb, dtype=torch.bool, device=device)
    total = n * nb
    for start in range(0, total, _CHUNK):
        stop = min(total, start + _CHUNK)
        idx = torch.arange(row0 * nb + start, row0 * nb + stop, dtype=torch.int64, device=device)
        out[start:stop] = uint32_at(seed, TID_MASK, 0, idx) < MASK_THRESHOLD
    return out.view(n, nb)


def tokens(seed: int, t: int, k: int, device="cpu") -> torch.Tensor:
    """x[t, k] bfloat16 ~ N(0, 1) (float32 sample rounded to nearest even)."""
    return normal(seed, TID_X, (t, k), 1.0, device).to(torch.bfloat16)


def logits(seed: int, t: int, e: int, device="cpu") -> torch.Tensor:
    """router logits[t, e] float32 ~ N(0, 1)."""
    return normal(seed, TID_LOGITS, (t, e), 1.0, device)


# The five decode-step workloads (the pages' shapes; config i uses seed i-1).
CONFIGS = {
    "linear_t1_k1024_n1024": dict(kind="linear", seed=0, t=1, k=1024, n=1024),
    "verify_t4_k7168_n7168": dict(kind="linear", seed=1, t=4, k=7168, n=7168),
    "lmhead_t4_k7168_n129280": dict(kind="linear", seed=2, t=4, k=7168, n=129280, x64=True),
    "ffn_up_k7168_n18432": dict(kind="linear", seed=3, t=(1, 2, 4, 8, 16, 32), k=7168, n=18432),
    "moe_e256_top8_t32": dict(kind="moe", seed=4, t=32, e=256, top_k=8, hidden=7168, inter=2048),
}
