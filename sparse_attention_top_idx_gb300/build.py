"""Build libdsaidx.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each .cu under csrc/ is compiled by nvcc in parallel and linked into
sparse_attention_top_idx_gb300/libdsaidx.so.  No cmake; a rebuild happens only
when a source or header is newer than the library.  build_peak() compiles the
tensor-core throughput probe (peak/mma_peak.cu) into libmmapeak.so, which the
benchmark uses as the denominator of the prefill roofline.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdsaidx.so")
PEAK_SRC = os.path.join(HERE, "peak", "mma_peak.cu")
PEAK_LIB = os.path.join(HERE, "libmmapeak.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, build_dir: str = BUILD, extra=()) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libdsaidx.so; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(_compile, srcs))
    if verbose:
        for _, log in results:
            print(log)
    tmp = LIB + ".tmp.%d" % os.getpid()
    # The driver entry point for TMA descriptors is looked up at run time
    # (cudaGetDriverEntryPointByVersion), so libcuda is not linked.
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


PHASES_LIB = os.path.join(HERE, "libdsaidx_phases.so")


def build_phases() -> str:
    """The diagnostic variant libdsaidx_phases.so: the same sources compiled
    with -DDSAIDX_PHASE_STAMPS (the decode kernel records %globaltimer at its
    phase boundaries).  Not part of the product build."""
    bdir = os.path.join(HERE, "_build_phases")
    if os.path.exists(PHASES_LIB) and all(os.path.getmtime(d) <= os.path.getmtime(PHASES_LIB) for d in _deps()):
        return PHASES_LIB
    os.makedirs(bdir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda src: _compile(src, bdir, ["-DDSAIDX_PHASE_STAMPS"]), srcs))
    tmp = PHASES_LIB + ".tmp.%d" % os.getpid()
    r = subprocess.run([nvcc()] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, PHASES_LIB)
    return PHASES_LIB


def build_peak(force: bool = False) -> str:
    """Compile and link libmmapeak.so (the tcgen05 throughput probe)."""
    deps = [PEAK_SRC, os.path.join(CSRC, "common.cuh"), os.path.abspath(__file__)]
    if not force and os.path.exists(PEAK_LIB) and all(os.path.getmtime(d) <= os.path.getmtime(PEAK_LIB) for d in deps):
        return PEAK_LIB
    tmp = PEAK_LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + ["-shared", PEAK_SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (PEAK_SRC, r.stdout, r.stderr))
    os.replace(tmp, PEAK_LIB)
    return PEAK_LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
    print(build_peak(force="--force" in sys.argv))
