"""Shared helpers for the GPU parity tests: inputs come from synth, expected
values from the oracle only, the outputs under test from the C ABI."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth


def lib():
    import mxfp4_weight_streaming_gb300 as mx
    mx.load()
    return mx


def bf16_to_f64(y: torch.Tensor) -> np.ndarray:
    return y.detach().float().cpu().numpy().astype(np.float64)


def sample_rows(n: int, count: int, seed: int = 0) -> np.ndarray:
    """Deterministic row sample: first/last rows, the tail row group, random rows."""
    rng = np.random.default_rng(seed)
    fixed = {0, 1, 15, 16, n - 1, n - 2, max(0, n - 17)}
    rand = rng.choice(n, size=min(n, count), replace=False)
    return np.array(sorted({int(r) for r in fixed if 0 <= r < n} | {int(r) for r in rand}), np.int64)


def assert_within(y_gpu: np.ndarray, y_ref: np.ndarray, rss: np.ndarray, what: str):
    ok = oracle.within_tolerance(y_gpu, y_ref, rss)
    if not ok.all():
        bad = np.argwhere(~ok)[:8]
        msgs = [f"{tuple(i)}: gpu={y_gpu[tuple(i)]!r} ref={y_ref[tuple(i)]!r} rss={rss[tuple(i)]!r}" for i in bad]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance\n" + "\n".join(msgs))


def linear_case(seed: int, t: int, k: int, n: int, x64: bool = False, device="cuda"):
    """(W float32 on device, x bf16 on device) for one dense workload."""
    w = synth.weights(seed, n, k, device=device, x64_blocks=x64)
    x = synth.tokens(seed, t, k, device=device)
    return w, x


GUARD_BYTES = 4096
CANARY = 0xA5


class Guarded:
    """A device tensor with GUARD_BYTES canary bytes on each side, so a test
    can check that a kernel wrote nothing outside the buffer it was given
    (the test-side stand-in for a memory checker). The tensor starts 4096
    bytes into a fresh allocation, so it keeps the allocator's alignment."""

    def __init__(self, shape, dtype, device="cuda"):
        shape = tuple(int(s) for s in shape)
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape, dtype=np.int64)) * itemsize
        self.raw = torch.full((2 * GUARD_BYTES + self.nbytes,), CANARY, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(shape)

    def check(self, what: str):
        torch.cuda.synchronize()
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        bad_h = int((head != CANARY).sum())
        bad_t = int((tail != CANARY).sum())
        assert bad_h == 0 and bad_t == 0, f"{what}: {bad_h} guard bytes before and {bad_t} after the buffer changed"
