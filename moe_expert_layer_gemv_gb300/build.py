"""Build libmoe_gb300.so (the C-ABI library of include/moe.h) in-tree for sm_103a.

One nvcc per translation unit, in parallel, then a shared link.  The -Xptxas -v
report (registers, spills, shared memory per kernel) goes to _build/ptxas.log.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_gb300.so")
SOURCES = ["api.cu", "route.cu", "expert_gemv.cu", "grouped_tc.cu", "tensor_map.cu", "combine.cu",
           "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
         "-Xptxas", "-v", f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}"]


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_gb300.so")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "moe.h"))
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append((s, o))
    nv = nvcc()
    logs = {}

    def compile_one(job):
        s, o = job
        r = subprocess.run([nv, *ARCH, *FLAGS, "-c", s, "-o", o], capture_output=True, text=True)
        return s, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for s, r in ex.map(compile_one, jobs):
                logs[s] = r.stdout + r.stderr
                if r.returncode != 0:
                    sys.stderr.write(logs[s])
                    raise RuntimeError(f"nvcc failed on {os.path.basename(s)}")
        with open(os.path.join(BUILD, "ptxas.log"), "a") as f:
            for s, text in logs.items():
                f.write(f"==== {os.path.basename(s)}\n{text}\n")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run([nv, *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
