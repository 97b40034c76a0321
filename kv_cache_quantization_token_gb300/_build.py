"""Builds libkvarn.so in-tree for sm_103a with nvcc (one translation unit per
kernel file, compiled in parallel, then linked with the static CUDA runtime)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libkvarn.so")
# (source, object, extra flags): decode.cu is built six times, for records
# with fp32 or binary16 scale fields and with 2-, 3- or 4-bit value codes.
UNITS = [("kvarn_abi.cu", "kvarn_abi.o", []), ("compress.cu", "compress.o", []),
         ("window.cu", "window.o", []), ("decode.cu", "decode.o", []),
         ("decode.cu", "decode_sb2.o", ["-DKVARN_BUILD_SCALE_BYTES=2"]),
         ("decode.cu", "decode_v4.o", ["-DKVARN_BUILD_V_BITS=4"]),
         ("decode.cu", "decode_sb2_v4.o", ["-DKVARN_BUILD_SCALE_BYTES=2", "-DKVARN_BUILD_V_BITS=4"]),
         ("decode.cu", "decode_v3.o", ["-DKVARN_BUILD_V_BITS=3"]),
         ("decode.cu", "decode_sb2_v3.o", ["-DKVARN_BUILD_SCALE_BYTES=2", "-DKVARN_BUILD_V_BITS=3"]),
         ("decode_noalloc.cu", "decode_noalloc.o", []), ("prefill.cu", "prefill.o", [])]
SOURCES = sorted({u[0] for u in UNITS})
HEADERS = [os.path.join(CSRC, "kvarn_common.cuh"), os.path.join(ROOT, "include", "kvarn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the KVarN CUDA library cannot be built")
    return path


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    objs, procs = [], []
    for src, obj, extra in UNITS:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, obj)
        objs.append(o)
        if force or _stale(o, [s] + HEADERS):
            cmd = [nvcc()] + ARCH + FLAGS + extra + ["-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd))
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"{src}:\n{out.decode(errors='replace')}")
    if errors:
        raise RuntimeError("nvcc failed\n" + "\n".join(errors))
    if force or _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        subprocess.run([nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs,
                       check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
