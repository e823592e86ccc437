"""Builds libfq.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu under csrc/ compiles to an object in parallel; the objects link into
fp8_dynamic_quant_gb300/libfq.so against the shared CUDA runtime.  Nothing is
installed outside this directory.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfq.so")
# engine-peak microbenchmarks for bench.py's roofline (not part of the fq ABI)
PEAKS_SRC = os.path.join(HERE, "peaks", "engine_peaks.cu")
PEAKS_LIB = os.path.join(HERE, "libfq_peaks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src, verbose):
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    return obj, r.stderr


def build_peaks(force=False):
    """Compile libfq_peaks.so (bench.py's engine microbenchmarks); returns its path."""
    deps = [PEAKS_SRC, os.path.join(CSRC, "fq_common.cuh"), __file__]
    if not force and os.path.exists(PEAKS_LIB):
        t = os.path.getmtime(PEAKS_LIB)
        if all(os.path.getmtime(d) < t for d in deps if os.path.exists(d)):
            return PEAKS_LIB
    tmp = PEAKS_LIB + ".tmp"
    cmd = [nvcc()] + ARCH + FLAGS + ["-shared", "-cudart", "shared", "-o", tmp, PEAKS_SRC,
                                     "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (PEAKS_SRC, r.stdout, r.stderr))
    os.replace(tmp, PEAKS_LIB)
    return PEAKS_LIB


def build(verbose=False, force=False):
    """Compile and link; returns the path of libfq.so."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + \
        [os.path.join(os.path.dirname(HERE), "include", "fq.h"), __file__]
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) < t for d in deps if os.path.exists(d)):
            return LIB
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        res = list(ex.map(lambda s: _compile(s, verbose), srcs))
    if verbose:
        for _, log in res:
            sys.stderr.write(log)
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + [o for o, _ in res] + \
        ["-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
