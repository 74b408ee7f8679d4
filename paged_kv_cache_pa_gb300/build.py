"""Build libpa_gb300.so in-tree with nvcc for sm_103a.

    python -m paged_kv_cache_pa_gb300.build [--force]

Every .cu file under csrc/ is compiled with nvcc and every .cpp file (host
code) with g++, in parallel, to _build/*.o, then linked into
paged_kv_cache_pa_gb300/libpa_gb300.so (CUDA runtime linked statically).
A stamp of the sources and flags skips the build when nothing changed.

build(variant="shortwait") makes a test copy, libpa_gb300_shortwait.so (objects
in _build_shortwait/), whose kernels give up their ordinary waits after a few
non-blocking polls; the tests use it to run the give-up path on the GPU.
build(variant="debug") makes libpa_gb300_debug.so (objects in _build_debug/):
the decode kernels check every work item and partition count they take
(PA_ERRBIT_INTERNAL), and every C-ABI compute call is an NVTX range.  The
product library is libpa_gb300.so.
"""
from __future__ import annotations

import glob
import hashlib
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpa_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                 "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


# variant -> (object folder, library, extra nvcc flags)
VARIANTS = {
    None: (BUILD, LIB, []),
    "shortwait": (os.path.join(ROOT, "_build_shortwait"),
                  os.path.join(PKG, "libpa_gb300_shortwait.so"), ["-DPA_TEST_WAIT_POLLS=4"]),
    "debug": (os.path.join(ROOT, "_build_debug"),
              os.path.join(PKG, "libpa_gb300_debug.so"), ["-DPA_DEBUG", "-DPA_NVTX"]),
}


def _stamp(sources, extra) -> str:
    h = hashlib.sha256()
    h.update(" ".join(CFLAGS + CXXFLAGS + extra).encode())
    for path in sorted(sources + glob.glob(os.path.join(CSRC, "*.cuh")) +
                       glob.glob(os.path.join(INCLUDE, "*.h"))):
        with open(path, "rb") as f:
            h.update(path.encode())
            h.update(f.read())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, variant=None) -> str:
    build_dir, lib, extra = VARIANTS[variant]
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    stamp = _stamp(sources, extra)
    stamp_file = lib + ".stamp"
    if (not force and os.path.exists(lib) and os.path.exists(stamp_file)
            and open(stamp_file).read() == stamp):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        if src.endswith(".cpp"):
            cmd = [os.environ.get("CXX", "g++")] + CXXFLAGS + ["-c", src, "-o", obj]
        else:
            cmd = [nvcc] + CFLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        results = list(ex.map(compile_one, sources))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
