"""Build the host (gcc) and device (nvcc, sm_103a) libraries of the input generator."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libsynth.so")
CUDA_LIB = os.path.join(HERE, "libsynth_cuda.so")


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t for s in sources)


def commands(cuda=True, force=False):
    """Compiler invocations still needed, as (argv, cwd) pairs."""
    cmds = []
    if force or _stale(HOST_LIB, ["synth.c", "synth.h"]):
        cmds.append((["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                      "-ffp-contract=off", "synth.c", "-o", HOST_LIB], HERE))
    if cuda and (force or _stale(CUDA_LIB, ["synth_cuda.cu", "synth.h"])):
        cmds.append((["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
                      "--fmad=false", "-Xcompiler", "-fPIC", "-shared", "synth_cuda.cu",
                      "-o", CUDA_LIB], HERE))
    return cmds


def build(cuda=True, force=False):
    procs = [subprocess.Popen(c, cwd=d) for c, d in commands(cuda, force)]
    for p in procs:
        if p.wait() != 0:
            raise RuntimeError(f"synth build failed: {p.args}")
