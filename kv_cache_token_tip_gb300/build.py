"""In-tree build of the CUDA libraries with nvcc (sm_103a).

``build()`` compiles every translation unit in parallel and links
``kv_cache_token_tip_gb300/libfasa.so`` (the FASA library) and
``workload/libfasa_synth.so`` (the synthetic-input generator used by the tests
and the benchmark).  Object files go to ``_build/`` at the repository root.
A library is rebuilt only when one of its sources is newer than it.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]

LIBFASA = os.path.join(PKG, "libfasa.so")
LIBSYNTH = os.path.join(ROOT, "workload", "libfasa_synth.so")

FASA_SOURCES = [os.path.join(PKG, "csrc", f) for f in
                ("fasa_api.cu", "fasa_cluster_bf16.cu", "fasa_cluster_f32.cu", "fasa_step_bf16.cu", "fasa_noalloc.cu",
                 "fasa_ca.cu")]
FASA_DEPS = [os.path.join(PKG, "csrc", f) for f in
             ("fasa_cluster.cuh", "fasa_step.cuh", "fasa_ptx.cuh", "fasa_internal.h")] + [
    os.path.join(ROOT, "include", "fasa.h")]
SYNTH_SOURCES = [os.path.join(ROOT, "workload", "csrc", "synth_gen.cu")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfasa")


def _stale(target, inputs) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(x) > t for x in inputs)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r


def _build_lib(target, sources, deps, extra_flags=(), verbose=False, force=False, ptxas_v=False):
    if not force and not _stale(target, sources + deps):
        return target
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    objs = []
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(sources), os.cpu_count() or 1))) as ex:
        for src in sources:
            obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
            objs.append(obj)
            cmd = [cc] + NVCC_FLAGS + list(extra_flags) + (["-Xptxas", "-v"] if ptxas_v else []) + [
                "-c", src, "-o", obj]
            jobs.append(ex.submit(_run, cmd, verbose))
        outs = [j.result() for j in jobs]
    if ptxas_v:
        for o in outs:
            print(o.stderr)
    tmp = target + ".tmp"
    _run([cc] + ARCH + ["-shared", "-o", tmp] + objs, verbose)
    os.replace(tmp, target)
    return target


def build(verbose=False, force=False, ptxas_v=False):
    """Compile libfasa.so and libfasa_synth.so (in parallel); return their paths."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        a = ex.submit(_build_lib, LIBFASA, FASA_SOURCES, FASA_DEPS, (), verbose, force, ptxas_v)
        b = ex.submit(_build_lib, LIBSYNTH, SYNTH_SOURCES, [], (), verbose, force, False)
        return a.result(), b.result()


if __name__ == "__main__":
    import sys
    print(build(verbose=True, force="--force" in sys.argv, ptxas_v="-v" in sys.argv))
