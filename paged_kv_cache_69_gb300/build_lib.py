"""Build libpa.so (the CUDA library behind include/pa.h) for sm_103a.

Each translation unit under csrc/ is compiled by its own nvcc process in
parallel, then linked into paged_kv_cache_69_gb300/libpa.so.  Rebuilds only
when a source or header is newer than the library.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libpa.so")
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"] + ARCH


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(ROOT, "include", "pa.h"), os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), csrc: str = None, out: str = None,
          build_dir: str = None) -> str:
    """Compile csrc/*.cu (or the given source folder) into libpa.so (or `out`)."""
    csrc = csrc or CSRC
    lib = out or LIB
    bdir = build_dir or BUILD
    if not force and lib == LIB and csrc == CSRC and up_to_date():
        return LIB
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = sorted(glob.glob(os.path.join(csrc, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


# ---------------------------------------------------------------------------
# host library (libpa_host.so: the block manager, plain C++, no CUDA)
# ---------------------------------------------------------------------------
HOST_SRC = os.path.join(HERE, "host")
HOST_LIB = os.path.join(HERE, "libpa_host.so")


def _host_deps():
    return sorted(glob.glob(os.path.join(HOST_SRC, "*.cpp"))) + \
        [os.path.join(ROOT, "include", "pa_block_manager.h"), os.path.abspath(__file__)]


def build_host(force: bool = False) -> str:
    """Compile host/*.cpp with the system C++ compiler into libpa_host.so."""
    if not force and os.path.exists(HOST_LIB) and \
            all(os.path.getmtime(d) <= os.path.getmtime(HOST_LIB) for d in _host_deps()):
        return HOST_LIB
    cxx = os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++")
    if not cxx:
        raise RuntimeError("no C++ compiler found")
    tmp = HOST_LIB + f".tmp{os.getpid()}"
    cmd = [cxx, "-O2", "-std=c++17", "-fPIC", "-shared", "-Wall", "-Wextra",
           *sorted(glob.glob(os.path.join(HOST_SRC, "*.cpp"))), "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"host build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, HOST_LIB)
    return HOST_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
    print(build_host(force="--force" in sys.argv))
