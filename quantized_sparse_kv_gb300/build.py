"""Build the kvq C-ABI shared library in-tree (nvcc, sm_103a).

``python -m quantized_sparse_kv_gb300.build`` compiles every ``csrc/*.cu`` to an
object file in parallel and links ``libkvq.so`` next to this file; with
``--debug`` it links ``libkvq_debug.so`` instead, the same sources compiled
with ``KVQ_DEBUG`` (every kernel checks each address range it derives from
its indices against the call's buffers and reports a miss as
KVQ_DEV_BOUNDS instead of making the access). It needs no GPU: nvcc
cross-compiles for sm_103a.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
OUT_DIR_DEBUG = os.path.join(PKG, "_build_debug")
LIB = os.path.join(PKG, "libkvq.so")
LIB_DEBUG = os.path.join(PKG, "libkvq_debug.so")
DEBUG_FLAGS = ["-DKVQ_DEBUG"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler",
         "-fvisibility=hidden", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def _compile(src: str, extra: list[str], out_dir: str) -> str:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def _link(objs: list[str], lib: str) -> str:
    cudalib = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath={cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def _variants(debug: bool | None):
    # (extra flags, object folder, library) of the release and/or debug build
    out = []
    if debug in (None, False):
        out.append(([], OUT_DIR, LIB))
    if debug in (None, True):
        out.append((DEBUG_FLAGS, OUT_DIR_DEBUG, LIB_DEBUG))
    return out


def build(verbose: bool = False, extra: list[str] | None = None,
          debug: bool | None = False) -> str:
    """Compile and link libkvq.so (debug=True: libkvq_debug.so; None: both,
    compiled in one pool). Returns the path of the release library, or of the
    debug one when only that was built."""
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = list(extra or [])
    jobs = []
    for flags, out_dir, lib in _variants(debug):
        os.makedirs(out_dir, exist_ok=True)
        jobs += [(src, extra + flags, out_dir) for src in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(16, len(jobs))) as ex:
        objs = list(ex.map(lambda j: _compile(*j), jobs))
    libs = []
    for i, (_, _, lib) in enumerate(_variants(debug)):
        libs.append(_link(objs[i * len(srcs):(i + 1) * len(srcs)], lib))
        if verbose:
            print(f"built {lib} from {len(srcs)} sources")
    return libs[0]


if __name__ == "__main__":
    args = sys.argv[1:]
    dbg = "--debug" in args
    build(verbose=True, extra=[a for a in args if a != "--debug"], debug=True if dbg else False)
