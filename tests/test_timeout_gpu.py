"""A bounded device wait that runs out, on a test-only build of the library.

Every wait in the kernels gives up after a time limit, sets the per-device
status word and lets the kernel wind down (no trap, no hang). Here a copy of
the library built with MXFP4_TEST_WITHHOLD_STAGE (never the product .so)
has CTA 0's producer withhold its first weight stage - no copy is issued and
no arrival made - and a 1 ms limit, so the consumers' wait on that stage
runs out. The call must report MXFP4_ERR_TIMEOUT through
mxfp4_last_device_status, leave the context usable, and the product library
must then give oracle-exact results. Cases: the streaming engine with lone
CTAs, and both tensor-core kernels (E4M3 split, packed E2M1) with lone CTAs
and with 2-CTA clusters (rank 0 times out while rank 1 hands it partials).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_within, bf16_to_f64, lib, linear_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def withhold_lib():
    from mxfp4_weight_streaming_gb300 import build
    path = build.build_test_variant("withhold", ["MXFP4_TEST_WITHHOLD_STAGE", "MXFP4_WAIT_LIMIT_NS=1000000ull"])
    L = ctypes.CDLL(path)
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    L.mxfp4_linear.restype = ctypes.c_int
    L.mxfp4_linear.argtypes = [P, I64, I64, P, P, I64, P, P]
    L.mxfp4_linear_plan.restype = ctypes.c_int
    L.mxfp4_last_device_status.restype = ctypes.c_int
    L.mxfp4_last_device_status.argtypes = [P]
    return L


@pytest.mark.parametrize("t,k,n,mode,cluster", [(2, 1056, 256, 0, 1), (20, 1024, 10240, 3, 1), (20, 4096, 256, 3, 2),
                                               (4, 1024, 20480, 4, 1), (4, 4096, 256, 4, 2), (12, 4096, 256, 4, 2)])
def test_bounded_wait_runs_out_and_context_survives(withhold_lib, t, k, n, mode, cluster):
    mx = lib()
    plan = mx.linear_plan(t, k, n)
    assert (plan["mode"], plan["cluster"]) == (mode, cluster), plan
    w, x = linear_case(130 + t, t, k, n)
    wq, ws = mx.quantize(w)
    stream = torch.cuda.current_stream().cuda_stream
    y = torch.zeros((t, n), dtype=torch.bfloat16, device="cuda")
    assert mx.last_device_status() == mx.MXFP4_OK
    rc = withhold_lib.mxfp4_linear(x.data_ptr(), t, k, wq.data_ptr(), ws.data_ptr(), n, y.data_ptr(), stream)
    assert rc == mx.MXFP4_OK  # the launch itself succeeds
    assert withhold_lib.mxfp4_last_device_status(stream) == mx.MXFP4_ERR_TIMEOUT
    assert withhold_lib.mxfp4_last_device_status(stream) == mx.MXFP4_OK  # read and cleared
    # The context is intact: the product library runs and matches the oracle.
    y2 = mx.linear(x, wq, ws)
    torch.cuda.synchronize()
    assert mx.last_device_status() == mx.MXFP4_OK
    rq, rs = oracle.quantize(w.cpu().numpy())
    y_ref, rss = oracle.linear(x, rq, rs)
    assert_within(bf16_to_f64(y2), y_ref, rss, f"after timeout t={t} k={k} n={n}")
