"""Build libxsattn.so (the sm_103a kernels + C ABI) in-tree with nvcc.

Three translation units are compiled in parallel and linked into one shared
library next to this file.  Only nvcc and the CUDA runtime are needed; no
PyTorch headers are involved (the C ABI takes plain pointers).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
SOURCES = ["attn_fwd.cu", "relayout.cu", "burst_gap.cu", "api.cu"]
HEADERS = ["kernels.h", "ptx.cuh", os.path.join("..", "..", "include", "xsattn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return os.path.join(cuda_home(), "bin", "nvcc")


# Library variants: the product library, and a build with per-tile timestamps
# (XS_TILE_SPANS; read by dit_attention_ulysses_gb300.spans) for measurements.
VARIANTS = {"": ([], "libxsattn.so", "_build"), "spans": (["-DXS_TILE_SPANS"], "libxsattn_spans.so", "_build_spans")}


def lib_path(variant: str = "") -> str:
    return os.path.join(HERE, VARIANTS[variant][1])


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [__file__]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    """Compile (if stale) and return the path of libxsattn.so (or of a variant)."""
    defines, lib_name, build_dir = VARIANTS[variant]
    LIB = os.path.join(HERE, lib_name)
    if not force and not _stale(LIB):
        return LIB
    bdir = os.path.join(HERE, build_dir)
    os.makedirs(bdir, exist_ok=True)
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-I", CSRC] + defines
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [_nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log:
                print(log)
    tmp = LIB + f".tmp{os.getpid()}"
    libdir = os.path.join(cuda_home(), "lib64")
    cmd = [_nvcc(), "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + [
        "--cudart", "shared", "-Xlinker", f"-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv, variant="spans" if "spans" in sys.argv else ""))
