"""mxfp4_moe_noalloc: the MoE entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the layer (plugins
whose framework's memory pool owns the device memory, serving loops that
forbid allocation after warm-up, loops that cannot take cudaMalloc's
implicit synchronisation). mxfp4_moe_noalloc keeps the layer's scratch in a fixed
array inside the library instead of a caller workspace. This file checks,
through the C ABI, that two calls in a row (the second one reusing the
array the first one left behind) give the same results as the workspace
entry point bit for bit and the oracle within the stated bound, and that
a problem too large for the array is refused. It is collected last so a
failure here does not hide any other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_cases import assert_within, bf16_to_f64, lib

pytestmark = pytest.mark.gpu


def _entry():
    L = lib().load()
    f = L.mxfp4_moe_noalloc
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.restype = I
    f.argtypes = [P, I64, I64, P, I64, I, P, P, P, P, I64, P, P, P, P]
    return f


def test_moe_noalloc_matches_workspace_entry_point_twice():
    """Two calls in a row through the C ABI. The second one has fewer tokens
    (fewer routed pairs) than the first, so it runs on the scratch contents
    the first call left behind. Each call's output must be within the stated
    bound of the oracle, and bit-identical (outputs, routing indices and gate
    weights) to the workspace entry point on the same inputs: the kernels
    are deterministic and only the scratch location differs."""
    mx = lib()
    noalloc = _entry()
    e, top_k, hidden, inter, seed = 64, 8, 1024, 512, 91
    w1 = synth.weights(seed, e * 2 * inter, hidden, device="cuda")
    w2 = synth.weights(seed, e * hidden, inter, tid=synth.TID_W2, device="cuda")
    w1q, w1s = mx.quantize(w1)
    w2q, w2s = mx.quantize(w2)
    r1q, r1s = oracle.quantize(w1.cpu().numpy())
    r2q, r2s = oracle.quantize(w2.cpu().numpy())
    W1 = {ex: (r1q.reshape(e, 2 * inter, -1)[ex], r1s.reshape(e, 2 * inter, -1)[ex]) for ex in range(e)}
    W2 = {ex: (r2q.reshape(e, hidden, -1)[ex], r2s.reshape(e, hidden, -1)[ex]) for ex in range(e)}
    dev = (w1q.view(e, 2 * inter, hidden // 2), w1s.view(e, 2 * inter, hidden // 32),
           w2q.view(e, hidden, inter // 2), w2s.view(e, hidden, inter // 32))
    stream = torch.cuda.current_stream().cuda_stream
    for call, t in enumerate((32, 19)):
        x = synth.tokens(seed + call, t, hidden, device="cuda")
        lg = synth.logits(seed + call, t, e, device="cuda")
        ids_ws = torch.empty((t, top_k), dtype=torch.int32, device="cuda")
        gw_ws = torch.empty((t, top_k), dtype=torch.float32, device="cuda")
        y_ws = mx.moe(x, lg, top_k, *dev, topk_ids=ids_ws, topk_w=gw_ws)
        ids_na = torch.empty((t, top_k), dtype=torch.int32, device="cuda")
        gw_na = torch.empty((t, top_k), dtype=torch.float32, device="cuda")
        y_na = torch.empty((t, hidden), dtype=torch.bfloat16, device="cuda")
        rc = noalloc(x.data_ptr(), t, hidden, lg.data_ptr(), e, top_k, dev[0].data_ptr(), dev[1].data_ptr(),
                     dev[2].data_ptr(), dev[3].data_ptr(), inter, y_na.data_ptr(), ids_na.data_ptr(),
                     gw_na.data_ptr(), stream)
        assert rc == mx.MXFP4_OK, mx.strerror(rc)
        torch.cuda.synchronize()
        lgn = lg.cpu().numpy()
        ids_ref, g_ref = oracle.route(lgn, top_k)
        assert np.array_equal(ids_na.cpu().numpy(), ids_ref)
        assert np.allclose(gw_na.cpu().numpy(), g_ref, rtol=1e-6, atol=0)
        y_ref, rss = oracle.moe(x, lgn, top_k, W1, W2, inter)
        assert_within(bf16_to_f64(y_na), y_ref, rss, f"no-alloc call {call + 1} (t={t})")
        assert torch.equal(ids_na, ids_ws)
        assert torch.equal(gw_na.view(torch.int32), gw_ws.view(torch.int32))
        assert torch.equal(y_na.view(torch.int16), y_ws.view(torch.int16)), f"call {call + 1}: differs from mxfp4_moe"
    assert mx.last_device_status() == mx.MXFP4_OK


def test_moe_noalloc_rejects_problems_larger_than_its_scratch():
    mx = lib()
    noalloc = _entry()
    t, e, top_k, hidden, inter = 256, 256, 16, 7168, 2048
    assert mx.mxfp4_moe_workspace_size(t, e, top_k, hidden, inter) > (12 << 20)
    p = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    rc = noalloc(p, t, hidden, p, e, top_k, p, p, p, p, inter, p, None, None, None)
    assert rc == mx.MXFP4_ERR_WORKSPACE
