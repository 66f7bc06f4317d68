"""Build synth/_build/libsynth.so, the device copy of the seeded input generator."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "_build", "libsynth.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def command():
    return [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared", "-Xcompiler",
            "-fPIC", "-Xcompiler", "-fvisibility=hidden", os.path.join(HERE, "synth_dev.cu"), "-o", OUT]


def build():
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    subprocess.run(command(), check=True)
    return OUT


if __name__ == "__main__":
    print(build())
