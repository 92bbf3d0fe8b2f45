"""Build the in-tree shared libraries for sm_103a with nvcc.

The translation units compile in parallel (one per input family plus the host
ABI), then link into ``block_scaled_grouped_gb300/_build/libbsgg.so`` with the
CUDA runtime linked statically.  ``debug_bounds=True`` builds the same sources
with -DBSGG_DEBUG_BOUNDS (every index range-checked on the device) into
``_build_debug/libbsgg_debug.so``.  No torch headers or libraries are involved.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libbsgg.so")
DEBUG_OUT_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_OUT_DIR, "libbsgg_debug.so")
_SHAPES = ["mxf8_128", "mxf8_256", "mxf8_pair", "nvf4_128", "nvf4_256", "nvf4_pair", "f4e8_128", "f4e8_256",
           "f4e8_pair"]
# forward and backward instances of each input family and tile shape in units
# of their own, so that they compile in parallel
UNITS = (["bsgg_host.cu", "bsgg_peak.cu"] + [f"bsgg_launch_{s}.cu" for s in _SHAPES] +
         [f"bsgg_launch_{s}_bwd.cu" for s in _SHAPES] + ["bsgg_launch_bf16_bwd.cu"])
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# hidden visibility (only the C ABI is exported) and no process-unique symbols:
# the release and the range-checking library share no internal symbol or
# function-local static when both are loaded
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-Xcompiler", "-fno-gnu-unique", "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbsgg")


def _sources_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "bsgg.h"), __file__]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    out_dir, lib_path = (DEBUG_OUT_DIR, DEBUG_LIB_PATH) if debug_bounds else (OUT_DIR, LIB_PATH)
    src_mtime = _sources_mtime()
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= src_mtime:
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    objs = []
    extra = ["-DBSGG_DEBUG_BOUNDS"] if debug_bounds else []

    def compile_unit(src: str) -> str:
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(compile_unit, UNITS))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    # the library carries the sources' time as the build found them: a source
    # edited while it compiled is newer, and the next call rebuilds
    os.utime(tmp, (src_mtime, src_mtime))
    os.replace(tmp, lib_path)
    return lib_path


def build_all(force: bool = False) -> None:
    """The release and the range-checking library, side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        for f in [ex.submit(build, force, False, dbg) for dbg in (False, True)]:
            f.result()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
