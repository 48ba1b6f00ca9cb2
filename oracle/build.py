"""Build the CPU oracle library (plain C, gcc, OpenMP, no FP contraction)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "liboracle.so")


def commands(force=False):
    src = os.path.join(HERE, "oracle.c")
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(src):
        return []
    return [(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
              "oracle.c", "-o", LIB, "-lm"], HERE)]


def build(force=False):
    for argv, cwd in commands(force):
        subprocess.check_call(argv, cwd=cwd)
