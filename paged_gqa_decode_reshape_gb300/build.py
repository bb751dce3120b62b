"""Build the CUDA library in-tree: paged_gqa_decode_reshape_gb300/_build/libpaged_decode.so.

Each .cu file under csrc/ is compiled for sm_103a in parallel, then linked
into one shared library with a static CUDA runtime. A second library,
libpaged_decode_faulttest.so, differs only in api.cu built with
-DPA_FAULT_TEST: it exports pa_fault_test_configure, with which the failure
tests make a kernel's bounded wait run out. Run with
``python -m paged_gqa_decode_reshape_gb300.build`` (add ``-v`` to print ptxas
register/spill reports).
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpaged_decode.so")
FAULT_LIB = os.path.join(BUILD, "libpaged_decode_faulttest.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(FAULT_LIB):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(FAULT_LIB))
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(job):
        src, suffix, defines = job
        obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", suffix + ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *defines, *extra, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, (r.stdout + r.stderr)

    srcs = _sources()
    api = os.path.join(CSRC, "api.cu")
    jobs = [(src, "", []) for src in srcs] + [(api, "_faulttest", ["-DPA_FAULT_TEST"])]
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose:
        for _, log in results[: len(srcs)]:
            sys.stdout.write(log)
    objs = [o for o, _ in results[: len(srcs)]]
    fault_objs = [results[-1][0] if o.endswith(os.sep + "api.o") else o for o in objs]

    def link(out, objects):
        tmp = out + f".{os.getpid()}.tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objects]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)

    link(LIB, objs)
    link(FAULT_LIB, fault_objs)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
