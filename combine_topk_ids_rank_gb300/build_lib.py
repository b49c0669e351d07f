"""Build libmoe_a2a.so in-tree for sm_103a with nvcc.

Translation units are compiled in parallel (one -gencode target), then
linked into a shared library next to this file.  Used by
__graft_entry__.build(); runnable as `python -m combine_topk_ids_rank_gb300.build_lib`.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(HERE, "libmoe_a2a.so")
BUILD_DIR = os.path.join(ROOT, "_build")
SOURCES = ["route.cu", "dispatch.cu", "combine.cu", "combine_ring.cu", "combine_small.cu", "combine_tree.cu",
           "dispatch_fp8.cu", "dispatch_small.cu", "dispatch_small_expert.cu", "route_expert.cu",
           "expert_gemm.cu", "expert_rank.cu",
           "moe_a2a.cpp", "moe_noalloc.cu"]
HEADERS = ["kernels.h", "expert.h", "dispatch_small.h", "smem_limit.h", "ptx.cuh", "fp8.cuh",
           "tcgen05.cuh", "f32x2.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _flags(verbose_ptxas: bool):
    f = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-O2",
         "-I" + INCLUDE, "-I" + CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "moe_a2a.h")]
    objs = []
    jobs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path, *headers]):
            lang = ["-x", "cu"] if src.endswith(".cu") else []
            jobs.append([nvcc(), *_flags(verbose_ptxas), *lang, "-c", path, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        return r.stdout + r.stderr

    logs = []
    if jobs:
        with ThreadPoolExecutor(len(jobs)) as pool:
            logs = list(pool.map(run, jobs))
    if force or jobs or _stale(LIBRARY, objs):
        tmp = LIBRARY + ".tmp%d" % os.getpid()
        cudalib = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")
        run([nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
             "-Xlinker", "-rpath," + cudalib])
        os.replace(tmp, LIBRARY)
    if verbose_ptxas:
        sys.stdout.write("".join(logs))
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
