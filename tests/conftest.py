import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


_PIN = None


def pin_library():
    """CUDA's host-side cuda_fp4.h conversions, built with g++ (test-only pin)."""
    global _PIN
    if _PIN is None:
        src = os.path.join(ROOT, "tests", "pins", "cuda_fp4_pin.cpp")
        out = os.path.join(ROOT, "tests", "pins", "libcudafp4pin.so")
        cuda_inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
        if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
            tmp = out + f".tmp{os.getpid()}"
            subprocess.check_call(["g++", "-O1", "-fPIC", "-shared", "-I", cuda_inc, src, "-o", tmp])
            os.replace(tmp, out)
        L = ctypes.CDLL(out)
        L.pin_e2m1_decode.restype = ctypes.c_float
        L.pin_e2m1_decode.argtypes = [ctypes.c_int]
        L.pin_e2m1_round.restype = ctypes.c_int
        L.pin_e2m1_round.argtypes = [ctypes.c_double]
        L.pin_e8m0_decode.restype = ctypes.c_float
        L.pin_e8m0_decode.argtypes = [ctypes.c_int]
        _PIN = L
    return _PIN


@pytest.fixture(scope="session")
def pin():
    return pin_library()


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()
