"""Build the CUDA library ``libfp8w8a8`` for sm_103a with nvcc.

One object per translation unit, compiled in parallel, then linked into a
shared library next to this file (``_build/libfp8w8a8_<machine>.so``).  The
CUDA runtime is linked statically, so the library loads on a machine without a
GPU (the host-side argument validation runs there); the driver is reached at
run time through the runtime.
"""
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["api.cu", "quant.cu", "gemm_decode.cu", "gemm_prefill.cu", "gemm_w8a16.cu"]
HEADERS = ["ptx.cuh", "kernels.h", "splitk.cuh", "norm_row.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--fmad=false", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return path


def lib_path() -> str:
    return os.path.join(BUILD_DIR, f"libfp8w8a8_{platform.machine()}.so")


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "fp8w8a8.h"),
                                                                  os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    out = lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= _newest_input():
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    mach = platform.machine()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, f"{os.path.splitext(src)[0]}_{mach}.o")
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
