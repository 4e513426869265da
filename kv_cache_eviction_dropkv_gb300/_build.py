"""Build step of the CUDA library: nvcc for sm_103a, in-tree output.

Compiles csrc/*.cu in parallel and links kv_cache_eviction_dropkv_gb300/_lib/libdropkv.so.
The library links the shared CUDA runtime (libcudart.so.13), so in a process
that imported torch first it shares torch's runtime and streams.

The "test_hooks" variant (libdropkv_test_hooks.so, -DDROPKV_TEST_HOOKS) is the
same source with the hooks of include/dropkv_test_hooks.h and a 10 ms pipeline
wait limit; only the tests build and load it.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(OUT_DIR, "libdropkv.so")
VARIANTS = {"": [], "test_hooks": ["-DDROPKV_TEST_HOOKS"]}
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-diag-suppress", "177"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libdropkv")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def lib_path(variant: str = "") -> str:
    return LIB_PATH if not variant else os.path.join(OUT_DIR, "libdropkv_%s.so" % variant)


def up_to_date(variant: str = "") -> bool:
    path = lib_path(variant)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build_library(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    path = lib_path(variant)
    if not force and up_to_date(variant):
        return path
    obj_dir = OUT_DIR if not variant else os.path.join(OUT_DIR, variant)
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    objs, procs = [], []
    for src in _sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *VARIANTS[variant], "-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join("%s\n%s" % f for f in failed))
    tmp = path + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path
