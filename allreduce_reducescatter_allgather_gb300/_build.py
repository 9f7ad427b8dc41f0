"""Compile the CUDA library (libvc.so) in-tree for sm_103a.

One nvcc process per translation unit, run in parallel, then one link.  The
library goes to ``_lib/libvc.so`` beside this file; objects and the ptxas
resource reports (registers, spills, stack) go to ``_build/``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIBDIR = PKG / "_lib"
LIB = LIBDIR / "libvc.so"

SOURCES = ["vc_api.cu", "vc_reduce_dispatch.cu", "vc_noalloc.cu", "vc_copy.cu", "vc_bucket.cu"]
HEADERS = ["vc_device.cuh", "vc_launch.cuh", "vc_bucket_kernel.cuh"]
# vc_reduce_inst.cu compiled once per (element type, op, order group):
# (object, -D flags).  Groups: 0 ring + recursive halving, 1 tree, 2 double
# binary tree.  The integer types have group 0 only (ring): their results
# do not depend on the order, so every order runs on the ring's kernels.
INSTANCE_SOURCE = "vc_reduce_inst.cu"
_TYPES = {"i32": "int32_t", "i64": "long long", "f32": "float", "bf16": "__nv_bfloat16"}
_OPS = {"sum": "OpSum", "prod": "OpProd", "max": "OpMax", "min": "OpMin"}
_GROUPS = (0, 1, 2)
INSTANCES = [(f"vc_reduce_{t}_{o}_g{g}", [f"-DVC_T={ct}", f"-DVC_OP={op}", f"-DVC_GROUP={g}",
                                          f"-DVC_FN=launch_reduce_{t}_{o}_g{g}"])
             for t, ct in _TYPES.items() for o, op in _OPS.items()
             for g in (_GROUPS if t in ("f32", "bf16") else (0,))]
# vc_bucket_inst.cu (the fused bucket AllReduce kernels) once per element type
BUCKET_SOURCE = "vc_bucket_inst.cu"
BUCKET_INSTANCES = [(f"vc_bucket_{t}", [f"-DVC_T={ct}", f"-DVC_FN=launch_bucket_{t}"])
                    for t, ct in _TYPES.items()]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libvc.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> Path:
    return Path(nvcc).resolve().parent.parent / "lib64"


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = [CSRC / s for s in SOURCES + HEADERS + [INSTANCE_SOURCE, BUCKET_SOURCE]] + [
        INCLUDE / "vc.h", Path(__file__)]
    return any(d.stat().st_mtime > t for d in deps)


def build_library(force: bool = False, jobs: int | None = None) -> Path:
    """Build libvc.so if it is missing or older than its sources."""
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    BUILD.mkdir(exist_ok=True)
    LIBDIR.mkdir(exist_ok=True)

    def compile_one(job):
        stem, src, defines = job
        obj = BUILD / (stem + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defines, "-I", str(INCLUDE), "-c", str(CSRC / src), "-o",
               str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        (BUILD / (stem + ".ptxas.log")).write_text(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {stem}:\n{r.stderr[-4000:]}")
        return obj

    jobs_list = [(Path(s).stem, s, []) for s in SOURCES]
    jobs_list += [(stem, INSTANCE_SOURCE, defs) for stem, defs in INSTANCES]
    jobs_list += [(stem, BUCKET_SOURCE, defs) for stem, defs in BUCKET_INSTANCES]
    # the longest units first (the bucket slices, then the double tree, tree
    # and ring slices, then the rest), so the pool finishes together
    jobs_list.sort(key=lambda j: -3 if j[1] == BUCKET_SOURCE
                   else (-int(j[0][-1]) if j[1] == INSTANCE_SOURCE else 1))
    jobs = jobs or max(1, os.cpu_count() or 4)
    with ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(compile_one, jobs_list))
    tmp = LIB.with_suffix(f".so.tmp{os.getpid()}")
    libdir = _cuda_lib_dir(nvcc)
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", str(tmp), *map(str, objs),
           "-Xlinker", f"-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True))
