"""Builds libpkv.so in-tree for sm_103a (GB300).

    python -m paged_kv_cache_152_gb300.build          # build if stale
    python -m paged_kv_cache_152_gb300.build --force  # rebuild everything

Every .cu file is compiled by nvcc with one -gencode (compute_103a ->
sm_103a), the host block manager by g++; translation units compile in
parallel and link into paged_kv_cache_152_gb300/libpkv.so (CUDA runtime linked
statically, so the library loads without LD_LIBRARY_PATH).
"""

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
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    cu = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    cpp = sorted(glob.glob(os.path.join(CSRC, "*.cpp")))
    deps = cu + cpp + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return cu, cpp, deps


def _stale(deps, lib=LIB):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force=False, verbose=False, ptxas_verbose=False, defines=(), lib_path=None):
    """Compile and link libpkv.so if any source changed; returns its path.

    defines (e.g. ["PKV_DECODE_G1_CUDACORE=1"]) and lib_path build a variant
    into another file (with its own object directory); a variant is rebuilt
    when a source is newer than it (its defines are the caller's to keep
    apart, one path per variant).
    """
    lib, obj_dir = LIB, OBJ
    if lib_path is not None:
        lib, obj_dir = os.path.abspath(lib_path), os.path.abspath(lib_path) + ".obj"
    cu, cpp, deps = _sources()
    if not force and not _stale(deps, lib):
        return lib
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC] + [f"-D{d}" for d in defines]
    jobs = []
    for src in cu:
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", *common, "-Xcompiler", "-fPIC", "-c", src, "-o", obj]
        if ptxas_verbose:
            cmd += ["-Xptxas", "-v"]
        jobs.append((cmd, obj))
    for src in cpp:
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        jobs.append((["g++", *common, "-fPIC", "-Wall", "-c", src, "-o", obj], obj))
    workers = min(len(jobs), max(2, os.cpu_count() or 2))
    logs = []
    with cf.ThreadPoolExecutor(workers) as ex:
        for out in ex.map(lambda j: _run(j[0]), jobs):
            logs.append(out)
    tmp = lib + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-Xcompiler", "-fPIC"])
    os.replace(tmp, lib)
    if verbose or ptxas_verbose:
        sys.stdout.write("".join(logs))
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas-v" in sys.argv)
    print(LIB)
