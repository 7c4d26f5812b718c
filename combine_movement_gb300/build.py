"""Build libep_gb300.so in-tree for sm_103a (nvcc, one -gencode, TUs compiled
in parallel, no cmake). ``python -m combine_movement_gb300.build`` or
``build()``; skipped when the library is newer than every source."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_objs")
LIB_PATH = os.path.join(PKG, "libep_gb300.so")

GENCODE = "arch=compute_103a,code=sm_103a"
NVCC_FLAGS = [
    "-O3", "-std=c++17", "-lineinfo", f"-gencode={GENCODE}",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills",
]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libep_gb300.so")
    return cand


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          out_dir: str | None = None) -> str:
    """Build the library; returns its path. With ``out_dir`` the objects and
    the library go there instead of in-tree (used to build the measured
    alternatives, e.g. ``extra_flags=["-DEP_COMBINE_MODE=1"]``, beside the
    default library)."""
    lib_path = os.path.join(out_dir, "libep_gb300.so") if out_dir else LIB_PATH
    obj_dir = os.path.join(out_dir, "_objs") if out_dir else OBJ_DIR
    if out_dir is None and not force and not is_stale():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(obj_dir, exist_ok=True)
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, "-shared", f"-gencode={GENCODE}", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
