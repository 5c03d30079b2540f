"""Build libpkv.so in-tree: nvcc for sm_103a, one job per translation unit, in parallel.

    python -m paged_kv_cache_278_gb300.build [--force] [--verbose]

The library lands next to this file (paged_kv_cache_278_gb300/libpkv.so) and
is rebuilt when any source under csrc/ or include/ is newer than it.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
import tempfile
import threading

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG_DIR, "libpkv.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]

_lock = threading.Lock()


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib_path: str = LIB_PATH) -> str:
    """Compile every csrc/ translation unit for sm_103a and link libpkv.so (or `lib_path`)."""
    with _lock:
        if not force and lib_path == LIB_PATH and not stale():
            return LIB_PATH
        nvcc = nvcc_path()
        tmp = tempfile.mkdtemp(prefix="pkv_build_")
        try:
            procs = []
            objs = []
            for src in sources():
                obj = os.path.join(tmp, os.path.basename(src) + ".o")
                cmd = [nvcc, *ARCH_FLAGS, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-c", src,
                       "-o", obj]
                if src.endswith(".cu") and verbose:
                    cmd += ["-Xptxas", "-v"]
                procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                                         text=True)))
                objs.append(obj)
            failed = []
            for src, cmd, p in procs:
                out, _ = p.communicate()
                if verbose or p.returncode != 0:
                    sys.stderr.write(f"$ {' '.join(cmd)}\n{out}")
                if p.returncode != 0:
                    failed.append(src)
            if failed:
                raise RuntimeError(f"nvcc failed for {failed}")
            out_tmp = os.path.join(tmp, "libpkv.so")
            link = [nvcc, *ARCH_FLAGS, "-shared", "-o", out_tmp, *objs, "-cudart", "static"]
            res = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
            if res.returncode != 0:
                sys.stderr.write(res.stdout)
                raise RuntimeError("link of libpkv.so failed")
            shutil.copy2(out_tmp, lib_path + f".tmp{os.getpid()}")
            os.replace(lib_path + f".tmp{os.getpid()}", lib_path)
        finally:
            shutil.rmtree(tmp, ignore_errors=True)
    return lib_path


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose))


if __name__ == "__main__":
    main()
