"""Build libcgtp.so in-tree: host C++ with g++, fixed kernels with nvcc for
sm_103a, the tensor-product kernel template embedded as a string for NVRTC.

Run ``python -m clebsch_gordan_tensor_gb300.build`` or call ``build()``.
Translation units compile in parallel; nothing is rebuilt when up to date.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libcgtp.so")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _embed(src: str, dst: str, symbol: str) -> None:
    with open(src) as f:
        text = f.read()
    delim = "CGTPSRC"
    assert f"){delim}\"" not in text
    body = f'namespace cgtp {{\nextern const char* {symbol};\nconst char* {symbol} = R"{delim}(' \
           f'{text}){delim}";\n}}\n'
    if not os.path.exists(dst) or open(dst).read() != body:
        with open(dst, "w") as f:
            f.write(body)


def _stale(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    inc = ["-I", os.path.join(ROOT, "include"), "-I", CSRC, "-I", os.path.join(CUDA, "include")]
    headers = [os.path.join(ROOT, "include", "cgtp.h"), os.path.join(CSRC, "plan.hpp"),
               os.path.join(CSRC, "internal.hpp"), os.path.join(CSRC, "tcgen05.cuh")]
    embed = os.path.join(OUT, "tp_kernels_embed.cpp")
    _embed(os.path.join(CSRC, "tp_kernels.cuh"), embed, "kTpKernelsSource")
    jobs = []
    for name in ("plan.cpp", "jit.cpp", "capi.cpp", "uvw.cpp"):
        src = os.path.join(CSRC, name)
        obj = os.path.join(OUT, name + ".o")
        cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-Wall", "-Wno-unused-function", *inc,
               "-c", src, "-o", obj]
        jobs.append((obj, [src, *headers], cmd))
    jobs.append((embed + ".o", [embed],
                 ["g++", "-std=c++17", "-O2", "-fPIC", "-c", embed, "-o", embed + ".o"]))
    for name in ("sh.cu", "graph.cu", "radial.cu", "linear.cu", "noalloc.cu", "probe.cu"):
        src = os.path.join(CSRC, name)
        obj = os.path.join(OUT, name + ".o")
        cmd = [os.path.join(CUDA, "bin", "nvcc"), *ARCH, "-std=c++17", "-O3", "-lineinfo",
               "-Xcompiler", "-fPIC", *inc, "-c", src, "-o", obj]
        jobs.append((obj, [src, *headers], cmd))

    def run(job):
        obj, deps, cmd = job
        if not _stale(obj, deps):
            return None
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            return f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
        return None

    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        errs = [e for e in ex.map(run, jobs) if e]
    if errs:
        raise RuntimeError("build failed:\n" + "\n".join(errs))
    objs = [j[0] for j in jobs]
    if _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = ["g++", "-shared", "-o", tmp, *objs, "-L", os.path.join(CUDA, "lib64"),
               "-lcudart", "-lnvrtc", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
