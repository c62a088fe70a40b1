"""Build libpq2.so, the CUDA library behind the C ABI of include/pq2.h.

Each translation unit under csrc/ is compiled by nvcc for sm_103a only, in
parallel, then linked into one shared library in this package directory.
build(debug=True) makes the bounds-checked library libpq2_debug.so instead
(PQ2_DEBUG=1: every kernel store checks its index against its buffer).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_objs")
LIB = os.path.join(HERE, "libpq2.so")
DEBUG_LIB = os.path.join(HERE, "libpq2_debug.so")
SOURCES = ["pq2_api.cu", "pq2_quant.cu", "pq2_gemv.cu", "pq2_small.cu", "pq2_tile.cu",
           "pq2_prefill.cu", "pq2_noalloc.cu", "pq2_bf16.cu", "pq2_multi.cu", "pq2_wtile.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the PQ2 CUDA library cannot be built")
    return cand


def _deps_mtime():
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(HERE, "..", "include", "pq2.h"))
    return max(os.path.getmtime(p) for p in paths if os.path.exists(p))


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    nvcc = _nvcc()
    out_dir = OUT_DIR + ("_debug" if debug else "")
    os.makedirs(out_dir, exist_ok=True)
    extra = ["-DPQ2_DEBUG=1"] if debug else []

    def compile_one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
