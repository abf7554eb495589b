"""Builds the seeded input generator (``gen.c``) into ``_gen.so`` beside it."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gen.c")
LIB = os.path.join(HERE, "_gen.so")


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
