"""Build libint8mp.so in-tree (int8_mixed_precision_row_gb300/_build/).

build(check=True) builds the bounds-checked variant (-DINT8MP_CHECK) into
_build_check/ instead: the same kernels with every computed global index
checked against its buffer (a failed check skips the access and is reported
as INT8MP_ERR_BOUNDS by int8mp_poll_device_status).

Each CUDA translation unit is compiled for sm_103a in parallel with nvcc and
the objects are linked into one shared library with the CUDA runtime linked
statically.  No fast-math: the quantizer's divisions, the epilogue's
multiplies and the bf16 rounding are IEEE round-to-nearest-even, and
subnormals are kept.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libint8mp.so")
CHECK_DIR = os.path.join(HERE, "_build_check")
CHECK_LIB = os.path.join(CHECK_DIR, "libint8mp.so")

SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "tma.cu", "noalloc.cu", "debug.cu"]
HEADERS = ["common.cuh", "ptx.cuh", "philox.cuh", "divide.cuh", "check.cuh", "codes.cuh"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + INCLUDE]


def _inputs():
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths += [os.path.join(INCLUDE, h) for h in ("int8mp.h", "int8mp_debug.h")]
    return paths + [os.path.abspath(__file__)]


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _compile(src: str, verbose: bool, out_dir: str = OUT_DIR, extra=()) -> str:
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, check: bool = False) -> str:
    out_dir, lib = (CHECK_DIR, CHECK_LIB) if check else (OUT_DIR, LIB)
    extra = ("-DINT8MP_CHECK",) if check else ()
    if not (force or stale(lib)):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, out_dir, extra), SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
