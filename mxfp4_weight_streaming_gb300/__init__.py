"""Thin Python binding of the MXFP4 weight-streaming C ABI (include/mxfp4.h).

Argument marshalling only: torch supplies device memory and the current CUDA
stream; every step of the computation runs in libmxfp4.so's kernels. There
is no CPU path: if the library has not been built, importing the C entry
points raises, and every compute call needs a CUDA device.

C entry points (same names as the header): mxfp4_quantize, mxfp4_linear,
mxfp4_linear_plan, mxfp4_moe, mxfp4_moe_workspace_size,
mxfp4_last_device_status, mxfp4_strerror. Convenience wrappers: quantize,
linear, linear_plan (host only), moe.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmxfp4.so")

MXFP4_OK = 0
MXFP4_ERR_INVALID_ARG = 1
MXFP4_ERR_SHAPE = 2
MXFP4_ERR_ALIGN = 3
MXFP4_ERR_WORKSPACE = 4
MXFP4_ERR_CUDA = 5
MXFP4_ERR_TIMEOUT = 6

EXPORTED = ["mxfp4_strerror", "mxfp4_quantize", "mxfp4_linear", "mxfp4_linear_plan", "mxfp4_moe_workspace_size",
            "mxfp4_moe", "mxfp4_last_device_status"]

_lib = None


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)}")
        self.status = status


class LinearPlan(ctypes.Structure):
    """mxfp4_linear_plan_t: how mxfp4_linear cuts the weight stream."""
    _fields_ = [(name, ctypes.c_int32) for name in ("mode", "ctas", "cluster", "stage_steps", "chunk_steps",
                                                     "ring_slots", "part_steps", "batch_units", "smem_bytes",
                                                     "group_rows")]


PLAN_MODES = {0: "whole K", 1: "K in parts", 2: "cluster split of K"}


def load() -> ctypes.CDLL:
    """Load libmxfp4.so (built by build.build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmxfp4.so is not built ({LIB_PATH}); run mxfp4_weight_streaming_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.mxfp4_strerror.restype = ctypes.c_char_p
    L.mxfp4_strerror.argtypes = [I]
    L.mxfp4_quantize.restype = I
    L.mxfp4_quantize.argtypes = [P, I64, I64, P, P, P]
    L.mxfp4_linear.restype = I
    L.mxfp4_linear.argtypes = [P, I64, I64, P, P, I64, P, P]
    L.mxfp4_moe_workspace_size.restype = ctypes.c_size_t
    L.mxfp4_moe_workspace_size.argtypes = [I64, I64, I, I64, I64]
    L.mxfp4_moe.restype = I
    L.mxfp4_moe.argtypes = [P, I64, I64, P, I64, I, P, P, P, P, I64, P, P, P, P, ctypes.c_size_t, P]
    L.mxfp4_moe_shared_workspace_size.restype = ctypes.c_size_t
    L.mxfp4_moe_shared_workspace_size.argtypes = [I64, I64, I, I, I64, I64]
    L.mxfp4_moe_shared.restype = I
    L.mxfp4_moe_shared.argtypes = [P, I64, I64, P, I64, I, I, P, P, P, P, I64, P, P, P, P, ctypes.c_size_t, P]
    L.mxfp4_ffn_workspace_size.restype = ctypes.c_size_t
    L.mxfp4_ffn_workspace_size.argtypes = [I64, I64, I64]
    L.mxfp4_ffn.restype = I
    L.mxfp4_ffn.argtypes = [P, I64, I64, P, P, P, P, I64, P, P, ctypes.c_size_t, P]
    L.mxfp4_last_device_status.restype = I
    L.mxfp4_last_device_status.argtypes = [P]
    L.mxfp4_linear_plan.restype = I
    L.mxfp4_linear_plan.argtypes = [I64, I64, I64, I, I, ctypes.POINTER(LinearPlan)]
    _lib = L
    return L


def strerror(status: int) -> str:
    return load().mxfp4_strerror(status).decode()


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, what: str):
    if rc != MXFP4_OK:
        raise Mxfp4Error(rc, what)


# ------------------------------------------------------- raw C entry points
def mxfp4_quantize(w_ptr, n, k, wq_ptr, ws_ptr, stream_ptr) -> int:
    return load().mxfp4_quantize(w_ptr, n, k, wq_ptr, ws_ptr, stream_ptr)


def mxfp4_linear(x_ptr, t, k, wq_ptr, ws_ptr, n, y_ptr, stream_ptr) -> int:
    return load().mxfp4_linear(x_ptr, t, k, wq_ptr, ws_ptr, n, y_ptr, stream_ptr)


def mxfp4_moe_workspace_size(t, e, top_k, hidden, inter) -> int:
    return load().mxfp4_moe_workspace_size(t, e, top_k, hidden, inter)


def mxfp4_moe(x_ptr, t, hidden, logits_ptr, e, top_k, w1q, w1s, w2q, w2s, inter, y_ptr, ids_ptr, gw_ptr,
              ws_ptr, ws_bytes, stream_ptr) -> int:
    return load().mxfp4_moe(x_ptr, t, hidden, logits_ptr, e, top_k, w1q, w1s, w2q, w2s, inter, y_ptr, ids_ptr,
                            gw_ptr, ws_ptr, ws_bytes, stream_ptr)


def mxfp4_moe_shared_workspace_size(t, e, top_k, n_shared, hidden, inter) -> int:
    return load().mxfp4_moe_shared_workspace_size(t, e, top_k, n_shared, hidden, inter)


def mxfp4_moe_shared(x_ptr, t, hidden, logits_ptr, e, top_k, n_shared, w1q, w1s, w2q, w2s, inter, y_ptr, ids_ptr,
                     gw_ptr, ws_ptr, ws_bytes, stream_ptr) -> int:
    return load().mxfp4_moe_shared(x_ptr, t, hidden, logits_ptr, e, top_k, n_shared, w1q, w1s, w2q, w2s, inter,
                                   y_ptr, ids_ptr, gw_ptr, ws_ptr, ws_bytes, stream_ptr)


def mxfp4_ffn_workspace_size(t, hidden, inter) -> int:
    return load().mxfp4_ffn_workspace_size(t, hidden, inter)


def mxfp4_ffn(x_ptr, t, hidden, w1q, w1s, w2q, w2s, inter, y_ptr, ws_ptr, ws_bytes, stream_ptr) -> int:
    return load().mxfp4_ffn(x_ptr, t, hidden, w1q, w1s, w2q, w2s, inter, y_ptr, ws_ptr, ws_bytes, stream_ptr)


def mxfp4_last_device_status(stream_ptr) -> int:
    return load().mxfp4_last_device_status(stream_ptr)


# ------------------------------------------------------ tensor wrappers
def quantize(w, stream=None):
    """float32 [n, k] CUDA tensor -> (wq uint8 [n, k/2], ws uint8 [n, k/32])."""
    import torch
    assert w.is_cuda and w.dtype == torch.float32 and w.dim() == 2 and w.is_contiguous()
    n, k = w.shape
    wq = torch.empty((n, k // 2), dtype=torch.uint8, device=w.device)
    ws = torch.empty((n, k // 32), dtype=torch.uint8, device=w.device)
    _check(mxfp4_quantize(w.data_ptr(), n, k, wq.data_ptr(), ws.data_ptr(), _stream(stream)), "mxfp4_quantize")
    return wq, ws


def linear(x, wq, ws, out=None, stream=None):
    """bf16 x [t, k] @ dequant(wq, ws)^T -> bf16 y [t, n]."""
    import torch
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    t, k = x.shape
    n = wq.shape[0]
    y = out if out is not None else torch.empty((t, n), dtype=torch.bfloat16, device=x.device)
    _check(mxfp4_linear(x.data_ptr(), t, k, wq.data_ptr(), ws.data_ptr(), n, y.data_ptr(), _stream(stream)),
           "mxfp4_linear")
    return y


def moe_workspace(t, e, top_k, hidden, inter, device, n_shared=0):
    import torch
    nbytes = mxfp4_moe_shared_workspace_size(t, e, top_k, n_shared, hidden, inter)
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def moe(x, logits, top_k, w1q, w1s, w2q, w2s, workspace=None, out=None, topk_ids=None, topk_w=None, stream=None,
        n_shared=0):
    """Grouped top-k MoE: x bf16 [t, hidden], logits f32 [t, e] -> bf16 [t, hidden].

    w1q/w1s: [e + n_shared, 2*inter, hidden/2] / [.., hidden/32] (gate rows first);
    w2q/w2s: [e + n_shared, hidden, inter/2] / [.., inter/32]. Experts e ..
    e + n_shared - 1 are shared experts every token applies with weight 1
    (mxfp4_moe_shared); n_shared = 0 calls mxfp4_moe.
    """
    import torch
    t, hidden = x.shape
    e = logits.shape[1]
    inter = w2q.shape[2] * 2
    if workspace is None:
        workspace = moe_workspace(t, e, top_k, hidden, inter, x.device, n_shared)
    y = out if out is not None else torch.empty((t, hidden), dtype=torch.bfloat16, device=x.device)
    ids_ptr = topk_ids.data_ptr() if topk_ids is not None else None
    gw_ptr = topk_w.data_ptr() if topk_w is not None else None
    if n_shared:
        _check(mxfp4_moe_shared(x.data_ptr(), t, hidden, logits.data_ptr(), e, top_k, n_shared, w1q.data_ptr(),
                                w1s.data_ptr(), w2q.data_ptr(), w2s.data_ptr(), inter, y.data_ptr(), ids_ptr, gw_ptr,
                                workspace.data_ptr(), workspace.numel(), _stream(stream)), "mxfp4_moe_shared")
    else:
        _check(mxfp4_moe(x.data_ptr(), t, hidden, logits.data_ptr(), e, top_k, w1q.data_ptr(), w1s.data_ptr(),
                         w2q.data_ptr(), w2s.data_ptr(), inter, y.data_ptr(), ids_ptr, gw_ptr, workspace.data_ptr(),
                         workspace.numel(), _stream(stream)), "mxfp4_moe")
    return y


def ffn(x, w1q, w1s, w2q, w2s, workspace=None, out=None, stream=None):
    """Fused dense FFN chain: bf16 x [t, hidden] -> bf16 W2 (SiLU(W1_gate x) * (W1_up x)) [t, hidden].

    w1q/w1s: [2*inter, hidden/2] / [2*inter, hidden/32] (gate rows first);
    w2q/w2s: [hidden, inter/2] / [hidden, inter/32].
    """
    import torch
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    t, hidden = x.shape
    inter = w2q.shape[1] * 2
    if workspace is None:
        workspace = torch.empty(mxfp4_ffn_workspace_size(t, hidden, inter), dtype=torch.uint8, device=x.device)
    y = out if out is not None else torch.empty((t, hidden), dtype=torch.bfloat16, device=x.device)
    _check(mxfp4_ffn(x.data_ptr(), t, hidden, w1q.data_ptr(), w1s.data_ptr(), w2q.data_ptr(), w2s.data_ptr(), inter,
                     y.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(stream)), "mxfp4_ffn")
    return y


def linear_plan(t, k, n, num_sms=152, max_smem=232448) -> dict:
    """The plan mxfp4_linear uses for this shape on a device with num_sms SMs
    and max_smem bytes of opt-in shared memory per block (GB300 defaults).
    Host only; raises Mxfp4Error when no plan fits."""
    plan = LinearPlan()
    _check(load().mxfp4_linear_plan(t, k, n, num_sms, max_smem, ctypes.byref(plan)), "mxfp4_linear_plan")
    return {name: getattr(plan, name) for name, _ in LinearPlan._fields_}


def last_device_status(stream=None) -> int:
    return mxfp4_last_device_status(_stream(stream))
