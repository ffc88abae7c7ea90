"""Build libdseq.so in-tree with nvcc for sm_103a.

Each .cu file under csrc/ compiles to an object under _build/ (in parallel),
then nvcc links them into libdseq.so next to this file.  The CUDA runtime is
linked statically and the driver API is reached through the runtime's entry
point query, so the library loads on a machine without a GPU driver (calls
then fail with DSEQ_ECUDA).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdseq.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["api.cu", "prep.cu", "ffma.cu", "tc_dseq.cu", "tc_bmu.cu", "gram.cu", "noalloc.cu",
           "som.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "dseq.h"))
    return files


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link libdseq.so if any source changed; return its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    deps = _deps()
    headers = [d for d in deps if not d.endswith(".cu")]
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        if force or _stale(obj, [s, *headers]):
            cmd = [nvcc, *NVCC_FLAGS, "-c", s, "-o", obj]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for out in ex.map(run, jobs):
                if (verbose or ptxas_info) and out:
                    print(out, file=sys.stderr)
    if force or jobs or _stale(LIB, objs):
        run([nvcc, *ARCH, "-shared", "-o", LIB, *objs])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
