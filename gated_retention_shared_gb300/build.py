"""Build libyoco.so (sm_103a) in-tree with nvcc.

Each translation unit compiles in parallel to an object, then one link step
makes gated_retention_shared_gb300/_build/libyoco.so.  Only sm_103a code is
generated.  Set YOCO_NVCC_EXTRA for extra flags (e.g. -Xptxas -v).
"""
import concurrent.futures as cf
import os
import shlex
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libyoco.so")
SOURCES = ["api.cu", "gret_simt.cu", "gret_tc.cu", "kv_proj.cu", "attn.cu", "attn_noalloc.cu", "kv_proj_tc.cu", "attn_tc.cu", "attn_fa.cu", "swa.cu", "gn_gate.cu", "rope.cu", "qkvg_tc.cu", "selftest.cu"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _flags():
    extra = shlex.split(os.environ.get("YOCO_NVCC_EXTRA", ""))
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC] + extra


def _compile(src):
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC, "-c", os.path.join(CSRC, src), "-o", obj] + _flags()
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose=False):
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    if verbose:
        for _, err in results:
            if err:
                print(err)
    objs = [o for o, _ in results]
    cmd = [NVCC, "-shared", "-o", LIB] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    subprocess.run(cmd, check=True)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv))
