"""Build libpaged_kv.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ compiles to an object in _build/ in
parallel; the objects link into paged_kv_cache_91_gb300/libpaged_kv.so against
the shared CUDA runtime, so the library and PyTorch share one runtime and one
primary context. ``python -m paged_kv_cache_91_gb300.build`` runs it.
"""
from __future__ import annotations

import glob
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpaged_kv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found")
    return p


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _stale(target: str, inputs) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib_path: str = LIB,
          build_dir: str = BUILD) -> str:
    """Compile what changed and link the library; returns its path.

    ``extra_flags`` (e.g. ``-DPKV_SIMT_RING_BYTES=65536``) with a separate
    ``lib_path``/``build_dir`` builds a tuning variant beside the default library.
    """
    BUILD_ = build_dir
    os.makedirs(BUILD_, exist_ok=True)
    stamp = os.path.join(BUILD_, "HOST_ARCH")
    arch = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != arch:
        force = True  # objects from another host architecture
    cc = nvcc()
    deps = _deps()
    srcs = _sources()
    objs = []
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD_, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + deps):
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        tmp = obj + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        log = os.path.join(BUILD_, os.path.basename(src) + ".log")
        with open(log, "w") as f:
            f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-6000:]}")
        os.replace(tmp, obj)
        return src

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src in ex.map(compile_one, jobs):
                if verbose:
                    print("compiled", os.path.relpath(src, ROOT), file=sys.stderr)
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-6000:]}")
        os.replace(tmp, lib_path)
        with open(stamp, "w") as f:
            f.write(arch + "\n")
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
