"""Builds the MSA CUDA library (libmsa.so) in-tree for sm_103a with nvcc.

Every translation unit under csrc/ is compiled in parallel (one -gencode, no cmake) and
linked into block_sparse_gqa_02_gb300/libmsa.so.  A stamp of the sources, headers and
flags skips the build when nothing changed.  The debug variant (-DMSA_DEBUG: device-side
index checks, see msa_debug_build in include/msa.h) builds the same sources into
libmsa_debug.so, in a build folder of its own.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmsa.so")
VARIANTS = {
    "release": (BUILD, LIB, []),
    "debug": (os.path.join(PKG, "_build_debug"), os.path.join(PKG, "libmsa_debug.so"),
              ["-DMSA_DEBUG"]),
}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the MSA CUDA library cannot be built")


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stamp(extra_flags) -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)) + ["../../include/msa.h"]:
        path = os.path.normpath(os.path.join(CSRC, name))
        if os.path.isfile(path):
            h.update(name.encode())
            with open(path, "rb") as f:
                h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()


def build(verbose: bool = False, extra_flags=(), force: bool = False,
          variant: str = "release") -> str:
    """Compile csrc/*.cu and link the library of `variant` ("release": libmsa.so, "debug":
    libmsa_debug.so); returns the library path."""
    build_dir, lib_path, variant_flags = VARIANTS[variant]
    extra_flags = list(variant_flags) + list(extra_flags)
    os.makedirs(build_dir, exist_ok=True)
    stamp_path = os.path.join(build_dir, "stamp")
    stamp = _stamp(extra_flags)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read() == stamp:
                return lib_path
    nvcc = _nvcc()
    flags = NVCC_FLAGS + list(extra_flags)

    def compile_one(src):
        obj = os.path.join(build_dir, src[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib_path


if __name__ == "__main__":
    args = sys.argv[1:]
    variant = "debug" if "--debug" in args else "release"
    extra = [a for a in args if a != "--debug"]
    print(build(verbose=True, extra_flags=extra, force=True, variant=variant))
