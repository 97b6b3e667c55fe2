"""The seeded input generator: exact integer hashing, determinism, distributions."""
import numpy as np
import torch

import synth


def test_mulmod32_exact():
    rng = np.random.default_rng(0)
    xs = rng.integers(0, 2 ** 32, 1000, dtype=np.uint64)
    for c in (0x7FEB352D, 0x846CA68B, 0xFFFFFFFF, 1):
        got = synth._mulmod32(torch.from_numpy(xs.astype(np.int64)), c).numpy()
        want = np.array([(int(v) * c) % 2 ** 32 for v in xs], dtype=np.int64)
        assert np.array_equal(got, want)


def test_hash_range_and_determinism():
    idx = torch.arange(0, 1 << 16, dtype=torch.int64)
    a = synth.uint32_at(1, 0, 0, idx)
    b = synth.uint32_at(1, 0, 0, idx)
    assert torch.equal(a, b)
    assert int(a.min()) >= 0 and int(a.max()) < 2 ** 32
    # different streams / tensors / seeds give different values
    assert not torch.equal(a, synth.uint32_at(1, 0, 1, idx))
    assert not torch.equal(a, synth.uint32_at(2, 0, 0, idx))
    # high index bits matter
    hi = synth.uint32_at(1, 0, 0, idx + (1 << 32))
    assert not torch.equal(a, hi)


def test_normal_moments_and_subrange():
    w = synth.weights(3, 512, 2048)
    assert w.dtype == torch.float32
    assert abs(float(w.mean())) < 2e-4
    assert abs(float(w.std()) - 0.02) < 2e-4
    part = synth.weights(3, 8, 2048, row0=100)
    assert torch.equal(part, w[100:108])


def test_tokens_are_bf16_rounded_normals():
    x = synth.tokens(0, 4, 4096)
    assert x.dtype == torch.bfloat16 and x.shape == (4, 4096)
    f = synth.normal(0, synth.TID_X, (4, 4096))
    assert torch.equal(x, f.to(torch.bfloat16))
    assert abs(float(x.float().std()) - 1.0) < 0.03


def test_x64_block_mask_rate():
    m = synth.block_x64_mask(2, 2000, 7168)
    rate = float(m.float().mean())
    assert 0.0085 < rate < 0.0115
    w = synth.weights(2, 40, 7168, x64_blocks=True)
    w0 = synth.weights(2, 40, 7168)
    mm = synth.block_x64_mask(2, 40, 7168).repeat_interleave(32, dim=1)
    assert torch.equal(w[mm], w0[mm] * 64) and torch.equal(w[~mm], w0[~mm])
