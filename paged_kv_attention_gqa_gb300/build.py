"""Build libpkv.so in-tree: nvcc for sm_103a, one process per translation unit.

    python -m paged_kv_attention_gqa_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
OUT = os.path.join(PKG, "libpkv.so")
OBJ = os.path.join(PKG, "_build")
SOURCES = ["pkv_api.cu", "decode.cu", "prefill.cu", "prefill_gather.cu", "prefill_pair.cu", "prefill_wide.cu",
           "planner.cpp"]
HEADERS = ["plan.h", "launch.h", "ptx.cuh", "tcgen05.cuh", "prefill_kernel.cuh", "prefill_pair.cuh",
           "prefill_wide.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(OBJ, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "pkv.h")]
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), *extra_flags]
    procs, objs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OBJ, src + ".o")
        objs.append(obj)
        if not force and not _stale(obj, [path, *hdrs]):
            continue
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, "-lineinfo", *common, "-c", path, "-o", obj]
            if verbose:
                cmd += ["-Xptxas", "-v"]
        else:
            cmd = [nvcc, *common, "-x", "c++", "-c", path, "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    if force or procs or _stale(OUT, objs):
        tmp = OUT + f".{os.getpid()}.tmp"
        subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"],
                       check=True)
        os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv)
    print(OUT)
