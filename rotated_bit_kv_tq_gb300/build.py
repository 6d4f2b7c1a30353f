"""Build the CUDA library libtq.so in-tree for sm_103a (nvcc, no CMake).

Each translation unit under csrc/ is compiled in parallel with relocatable device code
(the codebook tables and the device status word are shared across units), then nvcc
device-links and links them into rotated_bit_kv_tq_gb300/libtq.so.  Build products go
to rotated_bit_kv_tq_gb300/_build/ (git-ignored).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtq.so")
ROOT = os.path.dirname(HERE)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-rdc=true", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
           "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtq.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "tq.h")]


# The traced library (phase stamps of the decode-attention kernels, TQ_TRACE_PHASES), for
# bench.py --phase-trace; never loaded by the product path.
TRACE_BUILD = os.path.join(HERE, "_build_trace")
TRACE_LIB = os.path.join(HERE, "libtq_trace.so")


def _up_to_date(lib) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps() + [__file__])


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          trace: bool = False) -> str:
    out_lib, out_dir = (TRACE_LIB, TRACE_BUILD) if trace else (LIB, BUILD)
    if not force and not ptxas_info and _up_to_date(out_lib):
        return out_lib
    nvcc = _nvcc()
    os.makedirs(out_dir, exist_ok=True)
    objs = []
    jobs = []
    for src in _sources():
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVFLAGS, *(["-DTQ_TRACE_PHASES"] if trace else []), "-c", src, "-o", obj]
        if src.endswith(".cpp"):
            cmd[1:1] = ["-x", "cu"]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_info or r.returncode:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode:
                raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    tmp = out_lib + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-rdc=true", *objs, "-o", tmp]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(" ".join(link) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("nvcc link of libtq.so failed")
    os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_info="--ptxas" in sys.argv, trace="--trace" in sys.argv))
