"""Build ``libsp24.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel); the
objects are linked into one shared library with the CUDA runtime linked
statically, so the library loads without any other CUDA library on the path.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsp24.so")
SOURCES = ["sp24_abi.cu", "sp24_compress.cu", "sp24_gemm.cu", "sp24_gemm_pair.cu", "sp24_int8.cu"]
HEADERS = ["sp24_internal.cuh", "sp24_ptx.cuh", "sp24_gemm_common.cuh"]
ROOT = os.path.dirname(HERE)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-DSP24_BUILD", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "sp24.h"),
                                                                  os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    cmd = [_nvcc()] + ARCH + FLAGS + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile (if sources changed) and return the library path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


# A fault-test copy of the library for the tests of the give-up path: bounded
# waits give up after 1 ms, and the one-CTA GEMM kernel issues nothing for
# each CTA's first pipeline stage (SP24_FAULT_WITHHOLD_FIRST_STAGE), so that
# its MMA thread's wait runs out and the launch reports a device timeout.
# Built into _build/fault/, separate from libsp24.so, whose build never
# defines either macro.
FAULT_DIR = os.path.join(BUILD, "fault")
FAULT_LIB = os.path.join(FAULT_DIR, "libsp24_faulttest.so")
FAULT_FLAGS = ["-DSP24_WAIT_TIMEOUT_NS=1000000ull", "-DSP24_FAULT_WITHHOLD_FIRST_STAGE"]


def build_fault_test() -> str:
    """Compile (if sources changed) the fault-test library; return its path."""
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "sp24.h"),
                                                                  os.path.abspath(__file__)]
    if os.path.exists(FAULT_LIB) and all(os.path.getmtime(d) <= os.path.getmtime(FAULT_LIB) for d in deps):
        return FAULT_LIB
    os.makedirs(FAULT_DIR, exist_ok=True)

    def comp(src):
        obj = os.path.join(FAULT_DIR, src.replace(".cu", ".o"))
        cmd = [_nvcc()] + ARCH + FLAGS + FAULT_FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s" % (src, r.stderr))
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(comp, SOURCES))
    tmp = FAULT_LIB + ".tmp%d" % os.getpid()
    r = subprocess.run([_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stderr)
    os.replace(tmp, FAULT_LIB)
    return FAULT_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
