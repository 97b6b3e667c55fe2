"""The C-ABI library builds, loads on a machine without a GPU, exports every
function include/mxfp4.h declares, and rejects bad arguments before any
launch (these calls need no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mxfp4_weight_streaming_gb300 import build
    import mxfp4_weight_streaming_gb300 as mx
    build.build()
    return mx.load()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(mxfp4_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert "mxfp4_linear" in names and "mxfp4_moe" in names and "mxfp4_quantize" in names
    for name in names:
        assert hasattr(L, name), name


def test_only_the_c_abi_is_exported(L):
    """Every other symbol is private to the library: a process that loads two
    builds (a test variant beside the product) must not merge their launch
    caches, which gcc would otherwise emit as process-wide unique objects."""
    import shutil
    import subprocess
    import mxfp4_weight_streaming_gb300 as mx
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", mx.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines() if line.strip())
    assert exported == declared_functions()
    assert not [line for line in out.splitlines() if " u " in line]


def test_strerror(L):
    import mxfp4_weight_streaming_gb300 as mx
    for code in range(7):
        assert mx.strerror(code).startswith("MXFP4")
    assert "unknown" in mx.strerror(99)


def test_argument_errors_return_before_launch(L):
    import mxfp4_weight_streaming_gb300 as mx
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    odd = ctypes.c_void_p(0x1001)
    assert mx.mxfp4_linear(None, 1, 64, p, p, 8, p, None) == mx.MXFP4_ERR_INVALID_ARG
    assert mx.mxfp4_linear(p, 0, 64, p, p, 8, p, None) == mx.MXFP4_ERR_INVALID_ARG
    assert mx.mxfp4_linear(p, 1, 48, p, p, 8, p, None) == mx.MXFP4_ERR_SHAPE
    assert mx.mxfp4_linear(p, 33, 64, p, p, 8, p, None) == mx.MXFP4_ERR_SHAPE
    assert mx.mxfp4_linear(odd, 1, 64, p, p, 8, p, None) == mx.MXFP4_ERR_ALIGN
    assert mx.mxfp4_quantize(p, 4, 33, p, p, None) == mx.MXFP4_ERR_SHAPE
    assert mx.mxfp4_quantize(None, 4, 32, p, p, None) == mx.MXFP4_ERR_INVALID_ARG
    args = dict(t=4, hidden=64, e=8, top_k=2, inter=64)
    base = [p, args["t"], args["hidden"], p, args["e"], args["top_k"], p, p, p, p, args["inter"], p, None, None,
            p, 1 << 30, None]
    bad = list(base)
    bad[5] = 9  # top_k > e
    assert mx.mxfp4_moe(*bad) == mx.MXFP4_ERR_SHAPE
    bad = list(base)
    bad[14] = None  # no workspace
    assert mx.mxfp4_moe(*bad) == mx.MXFP4_ERR_WORKSPACE
    bad = list(base)
    bad[15] = 16  # workspace too small
    assert mx.mxfp4_moe(*bad) == mx.MXFP4_ERR_WORKSPACE
    bad = list(base)
    bad[2] = 48  # hidden % 32
    assert mx.mxfp4_moe(*bad) == mx.MXFP4_ERR_SHAPE
    assert mx.mxfp4_moe_workspace_size(32, 256, 8, 7168, 2048) > 0


def test_moe_shared_argument_errors_return_before_launch(L):
    import mxfp4_weight_streaming_gb300 as mx
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    t, hidden, e, top_k, inter = 4, 64, 8, 2, 64
    base = [p, t, hidden, p, e, top_k, 1, p, p, p, p, inter, p, None, None, p, 1 << 30, None]

    def call(**change):
        a = list(base)
        for i, v in change.items():
            a[int(i[1:])] = v
        return mx.mxfp4_moe_shared(*a)

    assert call(a6=-1) == mx.MXFP4_ERR_INVALID_ARG  # n_shared < 0
    assert call(a6=17) == mx.MXFP4_ERR_SHAPE  # n_shared > 16
    assert call(a4=1020, a6=5) == mx.MXFP4_ERR_SHAPE  # e + n_shared > 1024
    assert call(a15=None) == mx.MXFP4_ERR_WORKSPACE
    need = mx.mxfp4_moe_shared_workspace_size(t, e, top_k, 1, hidden, inter)
    assert need > mx.mxfp4_moe_workspace_size(t, e, top_k, hidden, inter)
    assert mx.mxfp4_moe_shared_workspace_size(t, e, top_k, 0, hidden, inter) == \
        mx.mxfp4_moe_workspace_size(t, e, top_k, hidden, inter)
    assert call(a16=need - 1) == mx.MXFP4_ERR_WORKSPACE
    assert mx.mxfp4_moe_shared_workspace_size(t, e, top_k, -1, hidden, inter) == 0


def test_ffn_argument_errors_return_before_launch(L):
    import mxfp4_weight_streaming_gb300 as mx
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    odd = ctypes.c_void_p(0x1001)
    base = [p, 4, 256, p, p, p, p, 128, p, p, 1 << 30, None]

    def call(**change):
        a = list(base)
        for i, v in change.items():
            a[int(i[1:])] = v
        return mx.mxfp4_ffn(*a)

    assert call(a0=None) == mx.MXFP4_ERR_INVALID_ARG
    assert call(a1=0) == mx.MXFP4_ERR_INVALID_ARG
    assert call(a1=9) == mx.MXFP4_ERR_SHAPE  # t > 8
    assert call(a2=48) == mx.MXFP4_ERR_SHAPE  # hidden % 32
    assert call(a7=80) == mx.MXFP4_ERR_SHAPE  # inter % 32
    assert call(a0=odd) == mx.MXFP4_ERR_ALIGN
    assert call(a9=None) == mx.MXFP4_ERR_WORKSPACE
    need = mx.mxfp4_ffn_workspace_size(4, 256, 128)
    assert need >= 256 + 4 * 128 * 4
    assert call(a10=need - 1) == mx.MXFP4_ERR_WORKSPACE
