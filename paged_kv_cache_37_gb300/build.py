"""In-tree build of libpagedkv.so for sm_103a.

Each translation unit of ``csrc/`` is compiled in parallel (nvcc for ``.cu``,
g++ for ``.cpp``), then linked with the static CUDA runtime so the library
loads on a machine without a GPU driver (the ABI test loads it on the CPU).
The driver API entry point the library needs (tensor-map encoding) is fetched
at run time through the runtime, so there is no link against libcuda.
"""
import glob
import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home():
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.exists(os.path.join(home, "bin", "nvcc")):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _sources():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    deps = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))
    return srcs, deps


def _stamp(srcs, deps, flags):
    h = hashlib.sha256()
    for f in srcs + deps:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def _compile(src, cuda, nvcc_flags, cxx_flags):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if src.endswith(".cu"):
        cmd = [os.path.join(cuda, "bin", "nvcc")] + nvcc_flags + ["-c", src, "-o", obj]
    else:
        cmd = ["g++"] + cxx_flags + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force=False, verbose=False):
    """Compile libpagedkv.so in-tree; skip when sources are unchanged."""
    cuda = _cuda_home()
    nvcc_flags = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                  "-I", INCLUDE, "--expt-relaxed-constexpr"] + ARCH
    if verbose:
        nvcc_flags += ["-Xptxas", "-v"]
    cxx_flags = ["-std=c++17", "-O2", "-fPIC", "-fvisibility=hidden", "-I", INCLUDE,
                 "-I", os.path.join(cuda, "include"), "-Wall"]
    srcs, deps = _sources()
    stamp = _stamp(srcs, deps, nvcc_flags + cxx_flags)
    stamp_file = os.path.join(BUILD, "stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return LIB
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda s: _compile(s, cuda, nvcc_flags, cxx_flags), srcs))
    if verbose:
        for _, log in results:
            if log:
                print(log)
    objs = [o for o, _ in results]
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [os.path.join(cuda, "bin", "nvcc"), "-shared", "--cudart", "static", "-o", tmp] + objs + ARCH
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
