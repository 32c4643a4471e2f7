"""Build the sm_103a shared library (libecho_gb300) in-tree with nvcc.

Each translation unit in csrc/ compiles in parallel to an object file under
_build/<machine>/, then one shared library is linked next to this file.  No
cmake, no torch extension machinery: the library has a plain C ABI
(include/echo.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build", platform.machine())
LIB_PATH = os.path.join(HERE, f"libecho_gb300_{platform.machine()}.so")
SOURCES = ["api.cu", "indexer.cu", "prefill.cu", "topk.cu", "cache_mgr.cu", "sparse_mla.cu", "validate.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                   "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib_path: str | None = None,
          build_dir: str | None = None) -> str:
    """Compile csrc/*.cu and link the shared library (default: the product build).
    `extra_flags`, `lib_path` and `build_dir` give a separate development build."""
    lib_out = lib_path or LIB_PATH
    bdir = build_dir or BUILD_DIR
    os.makedirs(bdir, exist_ok=True)
    hdrs = _headers()
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append((s, o))

    def compile_one(so):
        s, o = so
        cmd = [nvcc()] + _flags() + list(extra_flags) + ["-c", s, "-o", o + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(s)}:\n{r.stderr}")
        os.replace(o + ".tmp", o)
        log = os.path.join(bdir, os.path.basename(s) + ".ptxas.txt")
        with open(log, "w") as f:
            f.write(r.stderr)
        return r.stderr

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for out in ex.map(compile_one, jobs):
                if verbose:
                    print(out)
    if force or jobs or _stale(lib_out, objs):
        tmp = lib_out + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs + ["-lcudart_static", "-lrt", "-ldl", "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib_out)
    return lib_out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
