"""Build the C-ABI shared library ``libetattn.so`` in-tree with nvcc.

The library is compiled for sm_103a only.  The forward kernel source is
compiled once per (head dim, element type) variant so that the variants build
in parallel; the objects go to ``_build/`` at the repository root and the
library next to this file.  A stamp of the sources and flags skips rebuilds.

Usage: ``python -m exact_tiled_attention_19_gb300.build_lib [--force]``.
"""

from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libetattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
          "--expt-relaxed-constexpr", "-Xptxas", "-v"]
VARIANTS = [(d, bf) for d in (32, 64, 128) for bf in (0, 1)]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libetattn.so")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _stamp() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode() + b"\0" + f.read())
    h.update(" ".join(ARCH + CFLAGS).encode())
    return h.hexdigest()


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libetattn.so."""
    stamp = _stamp()
    stamp_file = os.path.join(BUILD_DIR, "stamp")
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = [([nvcc, *ARCH, *CFLAGS, "-c", os.path.join(CSRC, "attn_api.cu"), "-o",
              os.path.join(BUILD_DIR, "attn_api.o")], "attn_api"),
            ([nvcc, *ARCH, *CFLAGS, "-c", os.path.join(CSRC, "attn_combine.cu"), "-o",
              os.path.join(BUILD_DIR, "attn_combine.o")], "attn_combine")]
    jobs.append(([nvcc, *ARCH, *CFLAGS, "-c", os.path.join(CSRC, "attn_bwd_aux.cu"), "-o",
                  os.path.join(BUILD_DIR, "attn_bwd_aux.o")], "attn_bwd_aux"))
    for kind in ("fwd", "bwd"):
        for d, bf in VARIANTS:
            obj = os.path.join(BUILD_DIR, f"attn_{kind}_d{d}_{bf}.o")
            jobs.append(([nvcc, *ARCH, *CFLAGS, f"-DETATTN_INST_D={d}", f"-DETATTN_INST_BF16={bf}", "-c",
                          os.path.join(CSRC, f"attn_{kind}_inst.cu"), "-o", obj], f"{kind}_d{d}_{bf}"))
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(lambda j: (j[1], _run(j[0])), jobs))
    if verbose:
        for name, log in logs:
            print(f"== {name}\n{log}")
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        for name, log in logs:
            f.write(f"== {name}\n{log}\n")
    objs = [j[0][-1] for j in jobs]
    libdir = _cuda_lib_dir(nvcc)
    tmp = LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
          "-Xlinker", f"-rpath,{libdir}", "-L", libdir])
    os.replace(tmp, LIB_PATH)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
