"""Build libdspark.so for sm_103a with nvcc (in-tree, no CMake).

Each .cu under csrc/ compiles to an object in parallel, then the objects link
into ``_build/libdspark.so``.  The CUDA runtime is linked statically, so the
library depends only on the driver at run time.

``build(checked=True)`` makes the bounds-checked variant,
``_build/libdspark_checked.so``: the same sources compiled with
-DDSPARK_CHECKED, so that every index a kernel computes from data is tested
before the access (DSPARK_STATUS_OUT_OF_BOUNDS in include/dspark.h).  The
binding loads it instead of the normal library when the environment sets
DSPARK_CHECKED=1.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libdspark.so")
CHECKED_LIB_PATH = os.path.join(OUT_DIR, "libdspark_checked.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "plan.cu", "pack.cu", "accept.cu", "scatter.cu", "sample.cu", "calib.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdspark.so")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "dspark.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          checked: bool = False) -> str:
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    obj_dir = os.path.join(OUT_DIR, "checked") if checked else OUT_DIR
    os.makedirs(obj_dir, exist_ok=True)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _deps_mtime():
        return lib_path
    cc = nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", *ARCH_FLAGS, "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              *(["-DDSPARK_CHECKED"] if checked else []), *(extra_flags or [])]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [cc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
        return obj, p.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH_FLAGS, "-shared", "-o", tmp, *[o for o, _ in results]]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_all(force: bool = False) -> list[str]:
    """Both variants, compiled at the same time."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=2) as ex:
        futs = [ex.submit(build, force, False, None, checked) for checked in (False, True)]
        return [f.result() for f in futs]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))
