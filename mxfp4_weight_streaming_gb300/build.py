"""In-tree build of libmxfp4.so for sm_103a (nvcc, one -gencode, parallel TUs)."""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libmxfp4.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["quantize.cu", "linear.cu", "moe.cu", "capi.cu", "moe_noalloc.cu", "tc_linear.cu", "ffn.cu", "f4_linear.cu"]
NVCC = os.environ.get("NVCC", os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"))
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-gencode", "arch=compute_103a,code=sm_103a", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def _digest() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)) + [os.path.join("..", "..", "include", "mxfp4.h")]:
        path = os.path.normpath(os.path.join(CSRC, name))
        if os.path.isfile(path):
            h.update(name.encode())
            with open(path, "rb") as f:
                h.update(f.read())
    h.update(" ".join(FLAGS).encode())
    return h.hexdigest()[:16]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit and link libmxfp4.so; returns its path."""
    return _build(LIB, BUILD_DIR, [], force, verbose)


def build_test_variant(name: str, defines: list[str]) -> str:
    """A test-only copy of the library compiled with extra -D definitions,
    under _build/<name>/ (never the product libmxfp4.so); returns its path."""
    out_dir = os.path.join(BUILD_DIR, name)
    return _build(os.path.join(out_dir, f"libmxfp4_{name}.so"), out_dir, [f"-D{d}" for d in defines], False, False)


def _build(lib: str, build_dir: str, extra: list[str], force: bool, verbose: bool) -> str:
    os.makedirs(build_dir, exist_ok=True)
    stamp = os.path.join(build_dir, "stamp")
    digest = _digest() + " ".join(extra)
    if not force and os.path.exists(lib) and os.path.exists(stamp) and open(stamp).read() == digest:
        return lib

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [NVCC, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.append("-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
