"""Build libtfx_exl3.so in-tree for sm_103a with nvcc (no cmake).

Each bit width's kernels compile as their own object so the widths build in
parallel; the host side is one more object. The result lands next to this
file and is what the Python binding loads.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtfx_exl3.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags() -> list[str]:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                   "-I", INCLUDE, "-I", CSRC]


def _sources():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "tfx_exl3.h")]
    jobs = [(os.path.join(CSRC, "exl3_bits.cu"), os.path.join(OUT, f"exl3_b{b}.o"), [f"-DTFX_BITS={b}"])
            for b in range(1, 9)]
    jobs.append((os.path.join(CSRC, "exl3_host.cu"), os.path.join(OUT, "exl3_host.o"), []))
    jobs.append((os.path.join(CSRC, "exl3_noalloc.cu"), os.path.join(OUT, "exl3_noalloc.o"), []))
    jobs.append((os.path.join(CSRC, "exl3_encode.cu"), os.path.join(OUT, "exl3_encode.o"), []))
    return deps, jobs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    deps, jobs = _sources()
    nvcc = _nvcc()

    def compile_one(job):
        src, obj, extra = job
        if not force and not _stale(obj, deps):
            return obj, ""
        cmd = [nvcc, "-c", src, "-o", obj] + _flags() + extra + (["-Xptxas", "-v"] if ptxas_v else [])
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)} {extra}:\n{r.stderr[-4000:]}")
        return obj, r.stderr

    workers = min(len(jobs), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose:
        for obj, log in results:
            if log:
                print(f"== {os.path.basename(obj)}\n{log}")
    objs = [o for o, _ in results]
    if force or _stale(LIB, objs):
        cmd = [nvcc, "-shared", "-o", LIB + ".tmp"] + ARCH + objs + ["-cudart", "shared"]
        subprocess.run(cmd, check=True)
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_v="--ptxas-v" in sys.argv))
