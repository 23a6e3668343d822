"""Build ``libfp8norm.so`` (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled by nvcc in parallel, then linked into one
shared library next to this file.  Run ``python -m rmsnorm_fp8_activation_gb300.build``
or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfp8norm.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfp8norm")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return hs


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, variant: str | None = None,
          defines: tuple[str, ...] = ()) -> str:
    """Compile and link; returns the path of the shared library.

    variant: None builds the library (``libfp8norm.so`` next to this file);
    a name builds a test-only copy with the given preprocessor defines into
    ``_build/<name>/libfp8norm_<name>.so`` (e.g. the main pipeline waits
    limited to zero iterations, to run the timeout path)."""
    obj_dir = OBJ if variant is None else os.path.join(OBJ, variant)
    lib_path = LIB if variant is None else os.path.join(obj_dir, "libfp8norm_%s.so" % variant)
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE, "-I", CSRC] + ["-D" + d for d in defines]
    if verbose:
        common += ["-Xptxas", "-v"]
    hdrs = _deps()
    jobs = []
    for src in sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, [src] + hdrs):
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        tmp = obj + ".tmp%d" % os.getpid()
        r = subprocess.run([cc] + common + ["-c", src, "-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        os.replace(tmp, obj)
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for out in ex.map(compile_one, jobs):
            if verbose and out:
                print(out)
    objs = [os.path.join(obj_dir, os.path.basename(s)[:-3] + ".o") for s in sources()]
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp%d" % os.getpid()
        subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs, check=True)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
