"""Build libsnack.so (the CUDA library behind include/snack.h) in-tree.

Each ``csrc/*.cu`` compiles in parallel for sm_103a only, then links into
``_build/libsnack.so`` against the shared CUDA runtime (no other library).
A stamp keyed on the
sources, flags and host machine decides when to rebuild, so a library built
on another architecture is never reused.
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

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libsnack.so")
STAMP = os.path.join(BUILD, "libsnack.stamp")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = os.path.join(cuda, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _digest(extra_flags: list[str]) -> str:
    h = hashlib.sha256()
    for p in sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.hpp"))) + [
            os.path.join(INCLUDE, "snack.h")]:
        h.update(p.encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + extra_flags).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          out_dir: str | None = None) -> str:
    """Compile and link the library if needed; return its path.

    extra_flags (e.g. -D tuning macros) and out_dir build a separate copy
    without touching the default library."""
    extra_flags = list(extra_flags or [])
    build_dir = out_dir or BUILD
    lib_path = os.path.join(build_dir, "libsnack.so")
    stamp_path = os.path.join(build_dir, "libsnack.stamp")
    os.makedirs(build_dir, exist_ok=True)
    digest = _digest(extra_flags)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read().strip() == digest:
                return lib_path
    nv = nvcc()
    objs = []

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + f".{os.getpid()}.o")
        cmd = [nv, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = sources()
    planned = [os.path.join(build_dir, os.path.basename(src)[:-3] + f".{os.getpid()}.o") for src in srcs]
    tmp = lib_path + f".tmp{os.getpid()}"
    try:
        with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
            objs = list(ex.map(compile_one, srcs))
        cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nv)), "lib64")
        cmd = [nv, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath", "-Xlinker", cuda_lib]
        r = subprocess.run(cmd, capture_output=True, text=True)
    finally:  # no object file outlives the build, failed or not
        for o in planned:
            try:
                os.remove(o)
            except OSError:
                pass
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp_path, "w") as f:
        f.write(digest)
    return lib_path


PROBE_SRC = os.path.join(HERE, "probe", "gather_probe.cu")


def build_probe(force: bool = False) -> str:
    """Compile the gather-throughput probes (bench.py --gather-ceiling) into
    _build/libsnack_probe.so; not part of libsnack."""
    os.makedirs(BUILD, exist_ok=True)
    lib_path = os.path.join(BUILD, "libsnack_probe.so")
    stamp_path = os.path.join(BUILD, "libsnack_probe.stamp")
    h = hashlib.sha256()
    with open(PROBE_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    h.update(platform.machine().encode())
    digest = h.hexdigest()
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read().strip() == digest:
                return lib_path
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, "-shared", "-cudart", "shared", "-o", tmp, PROBE_SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on the probe:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp_path, "w") as f:
        f.write(digest)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
