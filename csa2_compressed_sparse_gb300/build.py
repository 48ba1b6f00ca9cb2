"""Build libcsa2.so (the C-ABI library) for sm_103a with nvcc.

Translation units are compiled in parallel and linked into one shared library next
to this file.  Only the CUDA toolkit is needed (no PyTorch extension machinery)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libcsa2.so")
SOURCES = ["csa2_api.cu", "k_compress.cu", "k_index.cu", "k_topk.cu", "k_attn.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "ptx.cuh", "compress_dev.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"] + ARCH


def _mtime(p):
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def objects():
    return [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]


def commands(force=False):
    """Compile commands still needed (as (argv, cwd) pairs); link is separate."""
    os.makedirs(BUILD, exist_ok=True)
    hdr = max(_mtime(os.path.join(CSRC, h)) for h in HEADERS)
    hdr = max(hdr, _mtime(os.path.join(HERE, "..", "include", "csa2.h")))
    cmds = []
    for s, o in zip(SOURCES, objects()):
        src = os.path.join(CSRC, s)
        if force or _mtime(o) < max(_mtime(src), hdr):
            cmds.append((["nvcc"] + FLAGS + ["-c", src, "-o", o], CSRC))
    return cmds


def link_command():
    return ["nvcc"] + ARCH + ["-shared", "--cudart", "static", "-o", LIB] + objects()


def needs_link():
    return _mtime(LIB) < max(_mtime(o) for o in objects())


def build(force=False, verbose=False):
    procs = []
    for argv, cwd in commands(force):
        procs.append(subprocess.Popen(argv, cwd=cwd, stdout=subprocess.PIPE,
                                      stderr=subprocess.STDOUT, text=True))
    logs = []
    for p in procs:
        out, _ = p.communicate()
        logs.append(out)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(p.args)}\n{out}")
    if needs_link():
        subprocess.check_call(link_command(), cwd=HERE)
    if verbose:
        print("\n".join(logs))
    return logs
