"""Builds libgdnspec.so in-tree with nvcc for sm_103a (no PyTorch extension
machinery; the library is plain C ABI and is loaded with ctypes)."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
# translation units: the decode / recurrent-prefill kernels with every C entry
# point, and the tensor-core chunked prefill
SRCS = [os.path.join(CSRC, "gdnspec.cu"), os.path.join(CSRC, "gdnprefill_chunked.cu")]
HEADERS = [os.path.join(ROOT, "include", "gdnspec.h"), os.path.join(CSRC, "gdn_internal.h")]
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD_DIR, "libgdnspec.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if a source or header is newer.  The translation
    units compile in parallel, then link into one shared library.  Returns its
    path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    newest = max(os.path.getmtime(f) for f in SRCS + HEADERS)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    tag = f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in SRCS:
        obj = os.path.join(BUILD_DIR, f"{os.path.splitext(os.path.basename(src))[0]}.{os.getpid()}.o")
        cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
    failed = []
    for src, proc in procs:
        out, err = proc.communicate()
        if proc.returncode != 0:
            sys.stderr.write(out + err)
            failed.append(os.path.basename(src))
        elif verbose:
            sys.stderr.write(err)
    if failed:
        raise RuntimeError(f"nvcc failed on {', '.join(failed)}")
    tmp = LIB + tag
    res = subprocess.run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs, "-o", tmp],
                         capture_output=True, text=True)
    for obj in objs:
        os.remove(obj)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed linking {LIB}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
