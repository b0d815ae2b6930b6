"""Build libkvq.so in-tree with nvcc for sm_103a (GB300).

Translation units compile in parallel; the CUDA runtime is linked statically so
the library loads beside any PyTorch build. Usage: ``python -m
bit_quantized_kv_append_gb300.build`` or ``build()`` from Python.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkvq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["kvq_api.cu", "kvq_rope.cu", "kvq_append.cu", "kvq_decode.cu", "kvq_levels.cu",
           "kvq_decode_b2.cu", "kvq_decode_b3.cu", "kvq_decode_b4.cu", "kvq_decode_b8.cu",
           "kvq_decode_tc_b2.cu", "kvq_decode_tc_b3.cu", "kvq_decode_tc_b4.cu",
           "kvq_decode_tc_b2o.cu", "kvq_decode_tc_b3o.cu", "kvq_decode_tc_b4o.cu",
           "kvq_decode_tc_b2p.cu", "kvq_decode_tc_b3p.cu", "kvq_decode_tc_b4p.cu",
           "kvq_decode_tc_b2op.cu", "kvq_decode_tc_b3op.cu", "kvq_decode_tc_b4op.cu",
           "kvq_decode_tc_b8.cu", "kvq_decode_tc_b8o.cu", "kvq_decode_tc_b8p.cu", "kvq_decode_tc_b8op.cu",
           "kvq_decode_tc_b2lv.cu", "kvq_decode_tc_b3lv.cu", "kvq_decode_tc_b4lv.cu", "kvq_decode_tc_b8lv.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "kvq.h")]
    return deps


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    out_dir = os.path.join(PKG, "_build")
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE,
             "--expt-relaxed-constexpr"]

    def compile_one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout, r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-shared", *ARCH, "-cudart", "static", *objs, "-o", tmp],
                       capture_output=True, text=True)
    if r.returncode:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
