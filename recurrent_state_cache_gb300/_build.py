"""Build of librsc.so: every .cu under csrc/ compiled for sm_103a, in parallel, then linked.

Only the sm_103a target is built (one -gencode).  The runtime is linked statically so
the library carries no dependency on a particular libcudart path.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "librsc.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a and link librsc.so; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in sources]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(sources), os.cpu_count() or 4)) as ex:
        list(ex.map(compile_one, zip(sources, objs)))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of librsc.so failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


WAIT_TEST_LIB = os.path.join(BUILD, "librsc_waittest.so")
WAIT_TEST_FLAGS = ["-DRSC_TEST_STARVE_FIRST_CHUNK", "-DRSC_MBAR_SPIN_LIMIT=65536u"]


def build_wait_test() -> str:
    """Test build of the decode path whose bounded wait runs out: decode.cu compiled with
    RSC_TEST_STARVE_FIRST_CHUNK (request 0's first state chunk is armed on its mbarrier but
    never copied) and a short spin limit, linked with the other objects of the library
    build.  Used only by the test of the give-up path; returns the library's path."""
    build()
    nvcc = _nvcc()
    src = os.path.join(CSRC, "decode.cu")
    obj = os.path.join(BUILD, "decode_waittest.o")
    r = subprocess.run([nvcc, *ARCH, *NVCC_FLAGS, *WAIT_TEST_FLAGS, "-c", src, "-o", obj],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on decode.cu (wait test):\n{r.stdout}\n{r.stderr}")
    others = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
              for s in sorted(glob.glob(os.path.join(CSRC, "*.cu")))
              if os.path.basename(s) != "decode.cu"]
    tmp = WAIT_TEST_LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, obj, *others], capture_output=True,
                       text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of the wait-test library failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, WAIT_TEST_LIB)
    return WAIT_TEST_LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
