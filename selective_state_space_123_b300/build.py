"""Build libssmscan.so in place (nvcc, sm_103a).

    python selective_state_space_123_b300/build.py [--force] [-j N]

(run as a script: importing the package itself needs the built library)

Each csrc/*.cu file is compiled to an object under _build/ (in parallel), then
linked into selective_state_space_123_b300/libssmscan.so.  Objects are rebuilt
when their source or any csrc header is newer.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libssmscan.so")
# register-only rate probes for the roofline (bench.py --workload peaks)
PROBE_SRC = os.path.join(CSRC, "probe", "ssm_peaks.cu")
PEAKS_LIB = os.path.join(PKG, "libssmpeaks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _compile(src: str, force: bool, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    newest_dep = max([os.path.getmtime(src)] + [os.path.getmtime(h) for h in _headers()])
    if force or not os.path.exists(obj) or os.path.getmtime(obj) < newest_dep:
        cmd = [nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj + ".tmp"]
        if verbose_ptxas:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose_ptxas:
            sys.stderr.write(r.stderr)
        os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, jobs: int = 0, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, force, verbose_ptxas), srcs))
    if force or not os.path.exists(LIB) or \
            os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
        os.replace(tmp, LIB)
    build_peaks(force)
    return LIB


def build_peaks(force: bool = False) -> str:
    deps = [PROBE_SRC] + _headers()
    if force or not os.path.exists(PEAKS_LIB) or \
            os.path.getmtime(PEAKS_LIB) < max(os.path.getmtime(d) for d in deps):
        tmp = PEAKS_LIB + ".tmp%d" % os.getpid()
        cmd = [nvcc(), *NVCC_FLAGS, "-shared", PROBE_SRC, "-o", tmp, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (PROBE_SRC, r.stdout, r.stderr))
        os.replace(tmp, PEAKS_LIB)
    return PEAKS_LIB


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-j", type=int, default=0)
    ap.add_argument("--ptxas-v", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, jobs=a.j, verbose_ptxas=a.ptxas_v))


if __name__ == "__main__":
    main()
