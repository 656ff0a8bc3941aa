"""Build libmq.so in-tree with nvcc for sm_103a (GB300).

One -gencode, translation units compiled in parallel, no cmake: quick enough
to run on the GPU host before tests.  No fast-math: the q8_0 quantizer's fp32
divisions must stay IEEE.  The result goes to quantized_decode_matvec_gb300/_lib/.
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
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libmq.so")

SOURCES = ["api.cu", "matvec.cu", "ffn.cu", "quantize.cu", "ring.cu", "step.cu", "noalloc.cu", "wtypes.cu", "ring_cols.cu", "ring_split.cu",
           "gemm.cu", "dequant.cu", "step_chained.cu", "mmq.cu"]
HEADERS = ["mq_device.cuh", "mq_stream.cuh", "mq_internal.h", "mq_job.cuh", "mq_epilogue.cuh", "mq_tma.cuh", "mq_unit.cuh", "mq_ring.cuh", "mq_ring_kernel.cuh", "mq_umma.cuh", "mq_step_kernel.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--extended-lambda", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "mq.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not needs_build():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for obj, err in ex.map(compile_one, SOURCES):
            objs.append(obj)
            if verbose and err:
                print(err, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    flags = [a for a in sys.argv[1:] if a.startswith("-X") or a.startswith("--")]
    print(build(force=True, verbose=True, extra_flags=[f for f in flags if f != "--force"]))
