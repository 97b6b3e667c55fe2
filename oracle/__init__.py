"""Python face of the MXFP4 CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. It wraps ``mxfp4_oracle.c``
(plain C, float64, OpenMP) through ctypes; ``build()`` compiles it with gcc.
Every array crosses as a contiguous numpy buffer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (gcc, -O2, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
                               "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(L):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    L.oracle_num_threads.restype = ctypes.c_int
    L.oracle_e2m1_value.restype = ctypes.c_double
    L.oracle_e2m1_value.argtypes = [ctypes.c_int]
    L.oracle_e8m0_value.restype = ctypes.c_double
    L.oracle_e8m0_value.argtypes = [ctypes.c_int]
    L.oracle_e2m1_round_magnitude.restype = ctypes.c_int
    L.oracle_e2m1_round_magnitude.argtypes = [ctypes.c_double]
    L.oracle_block_scale.restype = ctypes.c_int
    L.oracle_block_scale.argtypes = [P]
    L.oracle_quantize.restype = None
    L.oracle_quantize.argtypes = [P, I64, I64, P, P]
    L.oracle_dequant.restype = None
    L.oracle_dequant.argtypes = [P, P, I64, I64, P]
    L.oracle_linear.restype = None
    L.oracle_linear.argtypes = [P, I64, I64, P, P, I64, P, I64, P, P]
    L.oracle_route.restype = None
    L.oracle_route.argtypes = [P, I64, I64, ctypes.c_int, P, P]
    L.oracle_moe.restype = ctypes.c_int
    L.oracle_moe.argtypes = [P, I64, I64, P, I64, ctypes.c_int, ctypes.c_int, P, P, P, P, I64, P, I64, P, I64,
                              P, P]
    return L


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """bf16 bits as uint16 from a torch bfloat16 tensor or a uint16 array."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


class Oracle:
    """The oracle functions bound to one compiled copy of mxfp4_oracle.c."""

    def __init__(self, path: str):
        self.L = _bind(ctypes.CDLL(path))

    def num_threads(self) -> int:
        return self.L.oracle_num_threads()

    def e2m1_value(self, code: int) -> float:
        return self.L.oracle_e2m1_value(code)

    def e8m0_value(self, s: int) -> float:
        return self.L.oracle_e8m0_value(s)

    def e2m1_round_magnitude(self, a: float) -> int:
        return self.L.oracle_e2m1_round_magnitude(a)

    def block_scale(self, block: np.ndarray) -> int:
        b = np.ascontiguousarray(block, dtype=np.float32)
        assert b.size == 32
        return self.L.oracle_block_scale(_ptr(b))

    def quantize(self, w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
        """W float32 [n,k] -> (wq uint8 [n,k/2], ws uint8 [n,k/32])."""
        w = np.ascontiguousarray(w, dtype=np.float32)
        n, k = w.shape
        assert k % 32 == 0
        wq = np.empty((n, k // 2), np.uint8)
        ws = np.empty((n, k // 32), np.uint8)
        self.L.oracle_quantize(_ptr(w), n, k, _ptr(wq), _ptr(ws))
        return wq, ws

    def dequant(self, wq: np.ndarray, ws: np.ndarray) -> np.ndarray:
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        ws = np.ascontiguousarray(ws, dtype=np.uint8)
        n, kh = wq.shape
        out = np.empty((n, 2 * kh), np.float64)
        self.L.oracle_dequant(_ptr(wq), _ptr(ws), n, 2 * kh, _ptr(out))
        return out

    def linear(self, x, wq: np.ndarray, ws: np.ndarray, rows: np.ndarray | None = None):
        """Returns (y, rss) float64 [t, nrows] for the selected weight rows."""
        xb = _bf16_bits(x)
        t, k = xb.shape
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        ws = np.ascontiguousarray(ws, dtype=np.uint8)
        n = wq.shape[0]
        assert wq.shape[1] * 2 == k and ws.shape == (n, k // 32)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = n if rows is None else rows.size
        y = np.empty((t, nrows), np.float64)
        rss = np.empty((t, nrows), np.float64)
        self.L.oracle_linear(_ptr(xb), t, k, _ptr(wq), _ptr(ws), n, _ptr(rows), nrows, _ptr(y), _ptr(rss))
        return y, rss

    def route(self, logits: np.ndarray, top_k: int):
        """(ids int32 [t, top_k], g float64 [t, top_k])."""
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        t, e = lg.shape
        ids = np.empty((t, top_k), np.int32)
        g = np.empty((t, top_k), np.float64)
        self.L.oracle_route(_ptr(lg), t, e, top_k, _ptr(ids), _ptr(g))
        return ids, g

    def moe(self, x, logits: np.ndarray, top_k: int, w1: dict, w2: dict, inter: int,
            tok: np.ndarray | None = None, cols: np.ndarray | None = None, n_shared: int = 0):
        """Grouped top-k MoE in float64.

        ``w1``/``w2`` map expert id -> (wq, ws) packed arrays (only experts
        that the selected tokens route to are needed). With ``n_shared`` > 0,
        experts e .. e + n_shared - 1 (e = the logits' width) are shared
        experts that every token applies with weight 1. Returns (y, rss)
        float64 [ntok, ncols].
        """
        xb = _bf16_bits(x)
        t, hidden = xb.shape
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        e = lg.shape[1]
        arr = ctypes.c_void_p * max([e + n_shared] + [ex + 1 for ex in list(w1) + list(w2)])
        keep = []

        def table(d, idx):
            ptrs = arr()
            for ex, pair in d.items():
                a = np.ascontiguousarray(pair[idx], dtype=np.uint8)
                keep.append(a)
                ptrs[ex] = a.ctypes.data
            return ptrs

        p1q, p1s, p2q, p2s = table(w1, 0), table(w1, 1), table(w2, 0), table(w2, 1)
        if tok is not None:
            tok = np.ascontiguousarray(tok, dtype=np.int64)
        if cols is not None:
            cols = np.ascontiguousarray(cols, dtype=np.int64)
        ntok = t if tok is None else tok.size
        ncols = hidden if cols is None else cols.size
        y = np.empty((ntok, ncols), np.float64)
        rss = np.empty((ntok, ncols), np.float64)
        rc = self.L.oracle_moe(_ptr(xb), t, hidden, _ptr(lg), e, top_k, n_shared, p1q, p1s, p2q, p2s, inter,
                               _ptr(tok), ntok, _ptr(cols), ncols, _ptr(y), _ptr(rss))
        if rc != 0:
            raise ValueError("oracle_moe: a routed expert's weights were not provided")
        return y, rss


def default() -> Oracle:
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def num_threads() -> int:
    return default().num_threads()


def quantize(w):
    return default().quantize(w)


def dequant(wq, ws):
    return default().dequant(wq, ws)


def linear(x, wq, ws, rows=None):
    return default().linear(x, wq, ws, rows)


def route(logits, top_k):
    return default().route(logits, top_k)


def moe(x, logits, top_k, w1, w2, inter, tok=None, cols=None, n_shared=0):
    return default().moe(x, logits, top_k, w1, w2, inter, tok, cols, n_shared)


def ffn(x, w1q, w1s, w2q, w2s, inter, cols=None):
    """Dense SwiGLU FFN y = W2 (SiLU(W1_gate x) * (W1_up x)) in float64: the
    one-expert, top-1 MoE above (the softmax of a single logit is exactly 1,
    so its gate weight multiplies by 1). Returns (y, rss) [t, ncols]."""
    t = x.shape[0]
    lg = np.zeros((t, 1), np.float32)
    return default().moe(x, lg, 1, {0: (w1q, w1s)}, {0: (w2q, w2s)}, inter, cols=cols)


def within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, rss: np.ndarray,
                     rel: float = 4e-3, abs_rss: float = 1e-3) -> np.ndarray:
    """Elementwise |y - y_ref| <= rel*|y_ref| + abs_rss*rss (the stated bound)."""
    return np.abs(y_gpu.astype(np.float64) - y_ref) <= rel * np.abs(y_ref) + abs_rss * rss
