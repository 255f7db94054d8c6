"""In-tree build of libspecverify.so for sm_103a (nvcc, one translation unit).

The library links the CUDA runtime statically (nvcc's default), so it does not
depend on which libcudart the Python process has loaded; device pointers and
streams are shared through the driver's primary context.
"""

from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "spec_verify.cu")
OUT_DIR = os.path.join(PKG, "_lib")
OUT = os.path.join(OUT_DIR, "libspecverify.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path():
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if found:
        return found
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def build(verbose=False):
    os.makedirs(OUT_DIR, exist_ok=True)
    cmd = [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "--shared",
           "-Xcompiler", "-fPIC", "-Xptxas", "-v",
           "-I", os.path.join(ROOT, "include"), "-o", OUT, SRC]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(OUT_DIR, "build.log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stderr[-4000:])
    if verbose:
        print(res.stderr)
    return OUT


if __name__ == "__main__":
    print(build(verbose=True))
