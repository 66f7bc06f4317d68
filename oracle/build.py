"""Compile the CPU oracle (plain C, fp64) into oracle/_build/liboracle.so.

Test infrastructure: built by ``__graft_entry__.build()`` so the checker
exists on every machine; nothing in the CUDA library links it.
Floating-point contraction is off so x86 and Arm hosts give the same bits.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "_build", "liboracle.so")


def command():
    return ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", os.path.join(HERE, "oracle.c"), "-o", OUT, "-lm"]


def build():
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    subprocess.run(command(), check=True)
    return OUT


if __name__ == "__main__":
    print(build())
