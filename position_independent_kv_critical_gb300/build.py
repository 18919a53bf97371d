"""In-tree build of the C-ABI library ``_build/libpcf.so`` for sm_103a (GB300).

Two translation units compiled in parallel -- the host layout/RoPE code (g++) and the CUDA
kernels with their entry points (nvcc, ``-gencode arch=compute_103a,code=sm_103a``) -- then linked
into one shared library with the CUDA runtime linked statically.  No cmake, no torch extension
machinery: the library is plain C ABI.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT = os.path.join(HERE, "_build")
LIB_NAME = "libpcf.so"
GENCODE = "arch=compute_103a,code=sm_103a"


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if c and os.path.isdir(c):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("CUDA toolkit not found (set CUDA_HOME)")


def library_path() -> str:
    return os.path.join(OUT, LIB_NAME)


def _sources():
    files = []
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".cpp", ".h")):
                files.append(os.path.join(d, f))
    return files


def _digest() -> str:
    h = hashlib.sha256()
    h.update(GENCODE.encode())
    h.update(os.uname().machine.encode())
    for f in _sources():
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if the sources (or the machine architecture) changed; return its path."""
    os.makedirs(OUT, exist_ok=True)
    lib = library_path()
    stamp = os.path.join(OUT, "stamp.txt")
    digest = _digest()
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as fh:
            if fh.read().strip() == digest:
                return lib
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    tag = f"{os.getpid()}"
    host_o = os.path.join(OUT, f"pcf_host.{tag}.o")
    dev_o = os.path.join(OUT, f"pcf_device.{tag}.o")
    host_cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", os.path.join(cuda, "include"), "-c",
                os.path.join(CSRC, "pcf_host.cpp"), "-o", host_o]
    dev_cmd = [nvcc, "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "-Xptxas", "-v", "-c", os.path.join(CSRC, "pcf_device.cu"), "-o", dev_o]
    with concurrent.futures.ThreadPoolExecutor(2) as ex:
        fh = ex.submit(_run, host_cmd)
        fd = ex.submit(_run, dev_cmd)
        host_log, dev_log = fh.result(), fd.result()
    tmp = lib + f".{tag}.tmp"
    _run([nvcc, "-shared", "-cudart", "static", "-o", tmp, host_o, dev_o])
    os.replace(tmp, lib)
    for f in (host_o, dev_o):
        os.remove(f)
    with open(os.path.join(OUT, "ptxas.log"), "w") as fh_log:
        fh_log.write(dev_log)
    with open(stamp, "w") as fh_s:
        fh_s.write(digest)
    if verbose:
        sys.stdout.write(host_log + dev_log)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
