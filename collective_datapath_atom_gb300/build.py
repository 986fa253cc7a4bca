"""Build ``libpurlin.so`` in-tree for sm_103a (GB300) with nvcc.

Each translation unit is compiled in its own nvcc process, in parallel, then
linked into one shared library beside this file.  ``-Xptxas -v`` resource
reports go to ``_build/ptxas_<unit>.txt``.  The example kernels written
against the device-side API (``examples/``) are compiled in the same round
into ``libpurlin_examples.so``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpurlin.so")
BENCH = os.path.join(HERE, "purlin_bench")
EXAMPLES_DIR = os.path.join(HERE, "examples")
EXAMPLES_LIB = os.path.join(HERE, "libpurlin_examples.so")
SOURCES = ["plan.cpp", "api.cpp", "device_api.cpp", "channel_api.cpp", "vcounts_api.cpp", "kernels.cu",
           "kernels_ragged.cu", "noalloc.cu", "vcounts.cu", "packets.cu"]
EXAMPLE_SOURCES = ["device_examples.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpurlin.so")


def _stale() -> bool:
    outs = (LIB, BENCH, EXAMPLES_LIB)
    if not all(os.path.exists(o) for o in outs):
        return True
    t = min(os.path.getmtime(o) for o in outs)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps += [os.path.join(EXAMPLES_DIR, f) for f in os.listdir(EXAMPLES_DIR)]
    inc = os.path.join(HERE, "..", "include")
    deps += [os.path.join(inc, f) for f in os.listdir(inc)]
    deps.append(__file__)
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-I", os.path.join(HERE, "..", "include"), *ARCH]
    procs = []
    objs = []
    ex_objs = []
    units = [(CSRC, src, objs) for src in SOURCES] + \
            [(EXAMPLES_DIR, src, ex_objs) for src in EXAMPLE_SOURCES]
    for where, src, into in units:
        obj = os.path.join(BUILD, src.rsplit(".", 1)[0] + ".o")
        into.append(obj)
        cmd = [nvcc, *common, "-c", os.path.join(where, src), "-o", obj]
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        else:
            cmd = [nvcc, *common, "-x", "cu", "-c", os.path.join(where, src), "-o", obj]
        log = open(os.path.join(BUILD, f"ptxas_{src}.txt"), "w")
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for src, pr, log in procs:
        rc = pr.wait()
        log.close()
        if rc != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD, f"ptxas_{src}.txt")) as f:
                msgs.append(f"--- {src}\n" + f.read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    # the C benchmark program links the library through its public ABI
    tmp = BENCH + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, "-O2", "-I", os.path.join(HERE, "..", "include"),
                           os.path.join(CSRC, "purlin_bench.c"), "-o", tmp, "-L", HERE,
                           "-lpurlin", "-Xlinker", "-rpath,$ORIGIN", "-lm"])
    os.replace(tmp, BENCH)
    tmp = EXAMPLES_LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *ex_objs])
    os.replace(tmp, EXAMPLES_LIB)
    if verbose:
        with open(os.path.join(BUILD, "ptxas_kernels.cu.txt")) as f:
            sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
