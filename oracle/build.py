"""Builds the fp64 oracle (``mla_oracle.c``) into ``_oracle.so`` beside it.

Test infrastructure: the library is loaded only by the tests, the smoke check
and the benchmark's CPU-baseline leg.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mla_oracle.c")
LIB = os.path.join(HERE, "_oracle.so")


def command():
    return ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
            "-shared", SRC, "-o", LIB, "-lm"]


def needs_build():
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force=False):
    if force or needs_build():
        subprocess.run(command(), check=True)
    return LIB


if __name__ == "__main__":
    build(force=True)
    print(LIB)
