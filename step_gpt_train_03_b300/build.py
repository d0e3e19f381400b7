"""Build the CUDA library in-tree: step_gpt_train_03_b300/libgpt2_b300.so (sm_103a).

    python -m step_gpt_train_03_b300.build [--verbose-ptxas]
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgpt2_b300.so")
SOURCES = ["gpt2.cu", "gemm_tc.cu", "attention_tc.cu", "runtime.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _flags(ptxas_verbose=False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def build(ptxas_verbose=False, force=False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "gpt2.h")]
    newest = max(os.path.getmtime(d) for d in deps)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest and not ptxas_verbose:
        return LIB
    procs, objs = [], []
    for s in srcs:
        obj = os.path.join(BUILD, s.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [NVCC] + _flags(ptxas_verbose) + ["-c", os.path.join(CSRC, s), "-o", obj]
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if out.strip():
            print(f"--- {s}\n{out}", file=sys.stderr)
        if p.returncode != 0:
            failed.append(s)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    link = [NVCC] + ARCH + ["-shared", "-cudart", "shared", "-o", LIB] + objs
    subprocess.run(link, check=True)
    return LIB


if __name__ == "__main__":
    print(build(ptxas_verbose="--verbose-ptxas" in sys.argv, force=True))
