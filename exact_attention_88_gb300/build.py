"""In-tree build of libfa.so for sm_103a with nvcc (no cmake, no setuptools).

Each translation unit is compiled in parallel into `_build/`, then linked into
`libfa.so` next to this file.  Rebuilds only what changed; objects made on a
different host architecture are discarded first.

`libfa_diag.so` (from `csrc/diag/`) holds test-only diagnostics -- the
tensor-core operand-layout GEMM and the dropout-mask writer -- and links
against libfa.so; it is built beside it for the tests and is not part of
libfa's C ABI.
"""
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa.so")

SOURCES = [
    "fa_api.cu",
    "fa_fwd_sm103.cu",
    "fa_fwd64_sm103.cu",
    "fa_fwd128s_sm103.cu",
    "fa_bwd_sm103.cu",
    "fa_bwd_dkdv64_sm103.cu",
    "fa_bwd_dq64_sm103.cu",
    "fa_bwd_dq_sm103.cu",
    "fa_bwd_pair_sm103.cu",
    "fa_bwd_aux.cu",
    "fa_fp32.cu",
    "fa_probe.cu",
    "fa_noalloc.cu",
    "fa_tile_order.cu",
]
HEADERS = ["fa_common.cuh", "fa_internal.h", "fa_bwd_dkdv.cuh", "fa_bwd_dkdv64.cuh", "fa_bwd_dq.cuh",
           "fa_bwd_persist.cuh",
           "fa_bwd_dq64.cuh"]
DIAG_SOURCES = [os.path.join("diag", "fa_diag.cu")]
DIAG_LIB = os.path.join(HERE, "libfa_diag.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _newest_dep():
    paths = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "fa.h"), __file__]
    return max(os.path.getmtime(p) for p in paths)


def _compile(src, ptxas_verbose=False):
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    s = os.path.join(CSRC, src)
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(s), _newest_dep()):
        return obj, ""
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", s, "-o", obj]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return obj, r.stderr


def _link(lib, objs, deps, extra=()):
    newest = max(os.path.getmtime(p) for p in list(objs) + list(deps))
    if os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + list(objs) + list(extra)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)


def _host_stamp():
    return "%s %s" % (platform.machine(), platform.python_version())


def build(verbose=False, ptxas_verbose=False):
    """Compile every CUDA source for sm_103a and link libfa.so.  Returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "host.txt")
    old = open(stamp).read() if os.path.exists(stamp) else ""
    if old != _host_stamp():
        # objects or a library built on another host architecture: start over
        for f in os.listdir(BUILD):
            os.remove(os.path.join(BUILD, f))
        for lib in (LIB, DIAG_LIB):
            if os.path.exists(lib):
                os.remove(lib)
        with open(stamp, "w") as f:
            f.write(_host_stamp())
    every = SOURCES + DIAG_SOURCES
    with ThreadPoolExecutor(max_workers=min(len(every), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose), every))
    objs = [o for o, _ in results[:len(SOURCES)]]
    diag_objs = [o for o, _ in results[len(SOURCES):]]
    if verbose or ptxas_verbose:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    _link(LIB, objs, [])
    _link(DIAG_LIB, diag_objs, [LIB], extra=["-L", HERE, "-lfa", "-Xlinker", "-rpath=$ORIGIN"])
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
