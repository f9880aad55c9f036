"""Build libtq.so in-tree for sm_103a (nvcc + g++, translation units in parallel).

    python -m turboquant_compressed_kv_tq_gb300.build [--force] [-v]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libtq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["api.cu", "encode.cu", "encode_block.cu", "encode_tc.cu", "decode.cu", "decode_mma_a.cu", "decode_mma_b.cu", "decode_mma_c.cu", "decode_mma_d.cu", "decode_mma_e.cu", "decode_mma_f.cu", "decode_noalloc.cu", "decode_step.cu", "prefill_tc.cu", "cache_ops.cu", "decode_split.cu"]
CXX_SOURCES = ["codec_build.cpp"]
HEADERS = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))) + \
    [os.path.join(INCLUDE, "tq.h")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _commands():
    nvcc = _nvcc()
    cmds = []
    objs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        cmds.append((os.path.join(CSRC, src), obj,
                     [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE,
                      "-Xcompiler", "-fPIC,-ffp-contract=off", "-Xptxas", "-v" if _VERBOSE else "-O3",
                      "-c", os.path.join(CSRC, src), "-o", obj]))
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        cmds.append((os.path.join(CSRC, src), obj,
                     ["g++", "-O2", "-fPIC", "-std=c++17", "-ffp-contract=off", "-Wall", "-I", INCLUDE,
                      "-c", os.path.join(CSRC, src), "-o", obj]))
    return cmds, objs


_VERBOSE = False


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    global _VERBOSE
    _VERBOSE = verbose
    os.makedirs(BUILD, exist_ok=True)
    cmds, objs = _commands()
    procs = []
    for src, obj, cmd in cmds:
        if force or _stale(obj, [src, *HEADERS]):
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            sys.stdout.write(out.decode())
        if p.returncode != 0:
            failed.append((cmd, out.decode()))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("libtq build failed:\n" + msg)
    if force or procs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
