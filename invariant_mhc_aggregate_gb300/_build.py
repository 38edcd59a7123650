"""Compile the sm_103a library ``libmhc_h_aggregate.so`` in-tree with nvcc.

The library exports the C ABI of ``include/mhc_h_aggregate.h`` from
``csrc/mhc_h_aggregate.cu``; the kernels (``csrc/mhc_device.cuh``,
``csrc/mhc_coeffs.cuh``) are instantiated per storage type and coefficient
source in ``csrc/mhc_launch_*.cu``, compiled in parallel.  It is rebuilt when
its sources or flags change (a stamp file beside it records their hash).
"""

from __future__ import annotations

import hashlib
import os
import re
import shutil
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB_NAME = "libmhc_h_aggregate.so"
LIB_PATH = os.path.join(LIB_DIR, LIB_NAME)
SOURCES = [os.path.join(CSRC, f) for f in
           ("mhc_h_aggregate.cu", "mhc_launch_bf16.cu", "mhc_launch_f16.cu",
            "mhc_launch_sigmoid_bf16.cu", "mhc_launch_sigmoid_f16.cu", "mhc_launch_coeffs.cu",
            "mhc_launch_post.cu", "mhc_launch_post_sigmoid.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in
                  ("fastdiv.cuh", "mhc_coeffs.cuh", "mhc_device.cuh", "mhc_shift.cuh", "mhc_post.cuh",
                   "mhc_shift_bulk.cuh", "mhc_bulk.cuh", "mhc_f32x2.cuh", "mhc_launch.cuh", "mhc_launch_post.cuh")] \
    + [os.path.join(INCLUDE, "mhc_h_aggregate.h")]

ARCH = "sm_103a"

#: nvcc flags.  No fast math anywhere: the kernels promise IEEE round-to-nearest
#: binary32 products and sums, and subnormals kept.  ``--fmad=false`` keeps
#: nvcc from contracting a multiply and an add (the kernels use __fmul_rn /
#: __fadd_rn, which are never contracted, so this guards any code added later).
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "--fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", "-Xcompiler", "-fvisibility=hidden",
]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _digest(extra_flags) -> str:
    h = hashlib.sha256()
    for p in DEPS:
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()


def source_digest() -> str:
    """Hash of the library's sources and flags (identifies a library build)."""
    return _digest(())


KERNEL_FILES = [os.path.join(CSRC, f) for f in
                ("mhc_device.cuh", "mhc_coeffs.cuh", "mhc_shift.cuh", "mhc_shift_bulk.cuh", "mhc_post.cuh", "mhc_bulk.cuh",
                 "mhc_f32x2.cuh", "fastdiv.cuh", "mhc_launch.cuh", "mhc_launch_post.cuh", "mhc_launch_bf16.cu",
                 "mhc_launch_f16.cu", "mhc_launch_sigmoid_bf16.cu", "mhc_launch_sigmoid_f16.cu",
                 "mhc_launch_coeffs.cu", "mhc_launch_post.cu", "mhc_launch_post_sigmoid.cu")]


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace runs collapsed (string
    literals in these files hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_digest() -> str:
    """Hash of what decides the kernels' memory traffic: the device code, the
    launch shapes and the flags (not the host-side validation, and not the
    comments)."""
    h = hashlib.sha256()
    for p in KERNEL_FILES:
        with open(p) as f:
            h.update(_code_only(f.read()).encode())
    device_flags = []
    skip = False
    for flag in NVCC_FLAGS:            # host-compiler flags do not touch the kernels
        if skip:
            skip = False
        elif flag == "-Xcompiler":
            skip = True
        else:
            device_flags.append(flag)
    h.update(" ".join(device_flags).encode())
    return h.hexdigest()


def build(force: bool = False, extra_flags=(), verbose: bool = False) -> str:
    """Build the library if its sources or flags changed; return its path."""
    digest = _digest(extra_flags)
    stamp = LIB_PATH + ".stamp"
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = nvcc_path()
    with tempfile.TemporaryDirectory(dir=LIB_DIR) as work:
        # one translation unit per process, in parallel
        procs = []
        objs = []
        for src in SOURCES:
            obj = os.path.join(work, os.path.basename(src) + ".o")
            cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-c", "-o", obj, src]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                                text=True)))
            objs.append(obj)
        for cmd, proc in procs:
            out, err = proc.communicate()
            if proc.returncode != 0:
                raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{err}")
            if verbose and err:
                print(err)
        tmp = os.path.join(work, LIB_NAME)
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed ({' '.join(cmd)}):\n{res.stderr}")
        os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
