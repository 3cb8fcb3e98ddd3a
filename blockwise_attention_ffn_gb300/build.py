"""Builds libbpt.so (the CUDA library behind include/bpt.h) in-tree.

Every translation unit is compiled by nvcc for sm_103a in parallel, then
linked into one shared library with the CUDA runtime linked statically, so
loading the library needs only the NVIDIA driver (and nothing at all for
symbol inspection on a machine without a GPU)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libbpt.so")
SOURCES = ["bpt_api.cu", "gemm_tc.cu", "gemm_pair.cu", "attn_fwd.cu", "attn_bwd.cu", "attn_bwd_noalloc.cu", "norm_misc.cu",
           "host_util.cu", "lm_loss.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, obj: str, extra) -> None:
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
    if r.stderr.strip() and os.environ.get("BPT_BUILD_VERBOSE"):
        sys.stderr.write(r.stderr)


def build(force: bool = False, extra_flags=()) -> str:
    """Compile and link libbpt.so.  BPT_DEBUG=1 in the environment adds a
    short device-wait budget and a printf of the wait site on a timeout."""
    if os.environ.get("BPT_DEBUG") == "1":
        extra_flags = tuple(extra_flags) + ("-DBPT_WAIT_CYCLES=400000000LL", "-DBPT_TIMEOUT_PRINT")
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(HERE, "..", "include", "bpt.h"))
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= t for d in deps) and not extra_flags:
            return LIB
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)
    objs = [os.path.join(objdir, s.replace(".cu", ".o")) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(lambda so: _compile(so[0], so[1], list(extra_flags)), zip(SOURCES, objs)))
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    extra = sys.argv[1:]
    print(build(force=True, extra_flags=extra))
