"""Build libcbd.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel to an object in
_build/, then linked into continuous_batching_decode_gb300/libcbd.so (CUDA
runtime linked statically).  Objects are rebuilt when a source or header is
newer than them.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcbd.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I" + os.path.join(PKG, "..", "include")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _newest_header() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(PKG, "..", "include", "*.h"))
    return max(os.path.getmtime(h) for h in hs)


def build(verbose: bool = False, force: bool = False, extra: list | None = None, lib: str = LIB,
          build_dir: str = BUILD, src_dir: str = CSRC) -> str:
    """Compile and link; `extra` nvcc flags (e.g. -DCBD_TRACE for the
    timeline-tracing variant) or another `src_dir` go with `lib` /
    `build_dir` of their own."""
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(src_dir, "*.cu")) + glob.glob(os.path.join(src_dir, "*.cpp")))
    hdr = _newest_header()
    cc = nvcc()
    jobs = []
    for s in srcs:
        obj = os.path.join(build_dir, os.path.basename(s) + ".o")
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(s), hdr):
            cmd = [cc, *ARCH, *FLAGS, *(extra or []), "-c", s, "-o", obj]
            jobs.append((s, cmd))
    objs = [os.path.join(build_dir, os.path.basename(s) + ".o") for s in srcs]

    def run(job):
        s, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return s, cmd, r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for s, cmd, r in ex.map(run, jobs):
            if verbose or r.returncode:
                print(" ".join(cmd))
                print(r.stdout + r.stderr)
            if r.returncode:
                raise RuntimeError(f"nvcc failed on {os.path.basename(s)}")
    if jobs or force or not os.path.exists(lib):
        cmd = [cc, *ARCH, "-shared", "-o", lib, *objs, "-lcudart_static", "-ldl", "-lrt",
               "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            print(" ".join(cmd))
            print(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError("link of libcbd.so failed")
    return lib


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
