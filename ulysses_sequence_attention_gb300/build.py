"""Build libulysses.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled in parallel into ``_build/`` and linked into
``libulysses.so`` next to this file. The CUDA runtime is linked statically,
and the driver API is reached through ``cudaGetDriverEntryPointByVersion``, so
the library loads on a host without a GPU driver.

What is rebuilt follows content, not file times: each object records a key
(sha256 over its source, every header, the compiler flags, the compiler's
version and the host's machine type) in ``_build/<name>.key``, and the
library records the keys of the objects it was linked from. An object or a
library whose key differs from the current one, or is missing, is built
again, so a stale or foreign binary copied in beside the sources is never
reused.
"""
from __future__ import annotations

import concurrent.futures
import glob
import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libulysses.so")
INCLUDE = os.path.join(os.path.dirname(PKG_DIR), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-I" + INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _compiler_id(nvcc: str) -> str:
    p = subprocess.run([nvcc, "--version"], capture_output=True, text=True)
    return p.stdout.strip().splitlines()[-1] if p.returncode == 0 and p.stdout.strip() else nvcc


def _key(parts) -> str:
    h = hashlib.sha256()
    for part in parts:
        h.update(part if isinstance(part, bytes) else str(part).encode())
        h.update(b"\0")
    return h.hexdigest()


def _read(path: str) -> str:
    try:
        with open(path) as f:
            return f.read().strip()
    except OSError:
        return ""


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every kernel source and link the shared library. Returns its path."""
    srcs = _sources()
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = [_compiler_id(nvcc), platform.machine(), " ".join(NVCC_FLAGS)]
    common += [open(h, "rb").read() for h in _headers()]
    jobs, keys = [], {}
    for src in srcs:
        base = os.path.basename(src)[:-3]
        obj = os.path.join(BUILD_DIR, base + ".o")
        keys[src] = _key(common + [base, open(src, "rb").read(), ptxas_verbose])
        if force or not os.path.exists(obj) or _read(os.path.join(BUILD_DIR, base + ".key")) != keys[src]:
            cmd = [nvcc] + NVCC_FLAGS + (["-Xptxas", "-v"] if ptxas_verbose else []) + ["-c", src, "-o", obj]
            jobs.append((src, cmd))
    objs = [os.path.join(BUILD_DIR, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def run(job):
        src, cmd = job
        keyfile = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".key")
        if os.path.exists(keyfile):
            os.unlink(keyfile)      # no key for an object while it is being rewritten
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode == 0:
            with open(keyfile, "w") as f:
                f.write(keys[src])
        return src, p.returncode, p.stdout + p.stderr

    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src, rc, out in ex.map(run, jobs):
                if verbose or rc != 0 or ptxas_verbose:
                    sys.stderr.write(f"== {os.path.basename(src)}\n{out}")
                if rc != 0:
                    raise RuntimeError(f"nvcc failed on {src}")
    lib_key = _key([keys[s] for s in srcs] + [" ".join(ARCH)])
    lib_keyfile = os.path.join(BUILD_DIR, "libulysses.key")
    if force or jobs or not os.path.exists(LIB_PATH) or _read(lib_keyfile) != lib_key:
        tmp = LIB_PATH + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
        os.replace(tmp, LIB_PATH)
        with open(lib_keyfile, "w") as f:
            f.write(lib_key)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv)
    print(LIB_PATH)
