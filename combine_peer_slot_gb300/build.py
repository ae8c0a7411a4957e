"""Compile the CUDA library (sm_103a) into combine_peer_slot_gb300/libafd_gb300.so.

Each .cu translation unit is compiled in parallel with nvcc, then linked
into one shared library with the CUDA runtime linked statically.
build(debug=True) compiles the same sources with -DAFD_DEBUG_BOUNDS into
libafd_gb300_dbg.so: the kernels then check the indices they derive from
earlier kernels' outputs before using them (afd_debug_bounds in afd.h).
"""
import concurrent.futures as cf
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libafd_gb300.so")
OBJ_DBG = os.path.join(OBJ, "dbg")
LIB_DBG = os.path.join(HERE, "libafd_gb300_dbg.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]
SOURCES = ["afd_api.cu", "afd_kernels.cu", "afd_gemm_tc.cu", "afd_gemm_tc2.cu", "afd_noalloc.cu",
           "afd_attn.cu"]


def _compile(src, verbose, debug=False):
    out = os.path.join(OBJ_DBG if debug else OBJ, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *(["-DAFD_DEBUG_BOUNDS"] if debug else []), "-c",
           os.path.join(CSRC, src), "-o", out]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return out, r.stderr


def build(verbose=False, debug=False):
    os.makedirs(OBJ_DBG if debug else OBJ, exist_ok=True)
    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose, debug), SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    objs = [o for o, _ in results]
    lib = LIB_DBG if debug else LIB
    r = subprocess.run([NVCC, *ARCH, "-shared", "-o", lib, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


def needs_build(debug=False):
    lib = LIB_DBG if debug else LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "afd.h")]
    return any(os.path.getmtime(d) > t for d in deps)


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, debug="--debug" in sys.argv))
