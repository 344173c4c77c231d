"""Build liblinattn.so in-tree from csrc/*.cu for sm_103a.

One nvcc process per translation unit, run in parallel, then one link.
The library is linked against the shared CUDA runtime (libcudart.so.13), so
inside a process that already loaded PyTorch's runtime both use the same
one.  Nothing here needs a GPU: nvcc cross-compiles.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIBRARY = os.path.join(HERE, "liblinattn.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblinattn.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
                os.path.join("targets", "x86_64-linux", "lib")):
        p = os.path.join(root, sub)
        if os.path.isdir(p):
            return p
    return os.path.join(root, "lib64")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    files = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(INCLUDE, "*.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY):
        return False
    t = os.path.getmtime(LIBRARY)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: tuple[str, ...] = (),
          out: str | None = None) -> str:
    """Compile and link liblinattn.so unless it is already newer than its sources.

    `extra_flags` / `out` build a variant (e.g. an instrumented one) elsewhere."""
    target = out or LIBRARY
    if not force and out is None and up_to_date():
        return LIBRARY
    nvcc = _nvcc()
    flags = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
             "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "--expt-relaxed-constexpr",
             *extra_flags]
    objdir = tempfile.mkdtemp(prefix="linattn_build_")
    try:
        def compile_one(src):
            obj = os.path.join(objdir, os.path.basename(src) + ".o")
            cmd = [nvcc, *flags, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
            if verbose and r.stderr:
                sys.stderr.write(r.stderr)
            return obj

        with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
            objs = list(ex.map(compile_one, sources()))
        tmp_lib = os.path.join(objdir, "liblinattn.so")
        libdir = _cuda_lib_dir(nvcc)
        cmd = [nvcc, ARCH, "-shared", "-cudart", "shared", "-o", tmp_lib, *objs,
               "-Xlinker", f"-rpath={libdir}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp_lib, target)
    finally:
        shutil.rmtree(objdir, ignore_errors=True)
    return target


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
