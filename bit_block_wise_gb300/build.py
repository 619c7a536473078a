"""Build the CUDA library libbnb8.so in-tree (sm_103a only).

Each translation unit under csrc/ is compiled by nvcc in parallel, then
linked into a shared library next to this file.  Host code is compiled with
-ffp-contract=off and device code with --fmad=false, so every binary32
operation is rounded once in source order.
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbnb8.so")
# (source, object, extra flags): the step kernels compile once per optimizer
OPTIMIZERS = ["adam", "adamw", "momentum", "rmsprop", "adagrad", "lion", "ademamix"]
UNITS = [("bnb8_api.cu", "bnb8_api.o", []), ("k_quant.cu", "k_quant.o", [])] + [
    ("k_step_opt.cu", f"k_step_{name}.o", [f"-DBNB8_OPT={i}"]) for i, name in enumerate(OPTIMIZERS)]
SOURCES = sorted({src for src, _, _ in UNITS})
HEADERS = ["bnb8_internal.h", "bnb8_device.cuh", "k_step8.cuh", "k_step8_ring.cuh",
           "k_step8_ring_skip.cuh", "k_step32.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--fmad=false",
    "-Xcompiler", "-fPIC,-ffp-contract=off",
    "-I", os.path.join(ROOT, "include"), "-I", CSRC,
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "bnb8.h")]
    jobs = []
    for src, obj, extra in UNITS:
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ, obj)
        if force or ptxas_info or _stale(o, [s] + hdrs):
            cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", s, "-o", o]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append((obj, cmd))
    outputs = {}
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            futs = {ex.submit(subprocess.run, cmd, capture_output=True, text=True): src
                    for src, cmd in jobs}
            for f in concurrent.futures.as_completed(futs):
                r = f.result()
                outputs[futs[f]] = r.stderr + r.stdout
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed for {futs[f]}:\n{r.stderr}{r.stdout}")
    objs = [os.path.join(OBJ, obj) for _, obj, _ in UNITS]
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}{r.stdout}")
        os.replace(tmp, LIB)
    if verbose or ptxas_info:
        for src, out in sorted(outputs.items()):
            if out.strip():
                print(f"== {src}\n{out}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
