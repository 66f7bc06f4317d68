"""Build libyoco.so (sm_103a) in-tree with nvcc.

Each translation unit compiles in parallel to an object, then one link step
makes gated_retention_shared_gb300/_build/libyoco.so.  Only sm_103a code is
generated.  Set YOCO_NVCC_EXTRA for extra flags (e.g. -Xptxas -v).

build(debug=True) makes _build_debug/libyoco.so instead, compiled with
YOCO_DEBUG_CHECKS: every kernel checks the indices it forms before using them
and records a failed check for yoco_debug_checks (never a trap).
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
DEBUG_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB = os.path.join(DEBUG_DIR, "libyoco.so")
SOURCES = ["api.cu", "gret_simt.cu", "gret_tc.cu", "kv_proj.cu", "attn.cu", "attn_noalloc.cu", "kv_proj_tc.cu", "attn_tc.cu", "attn_fa.cu", "swa.cu", "gn_gate.cu", "rope.cu", "qkvg_tc.cu", "selftest.cu"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _flags(debug=False):
    extra = shlex.split(os.environ.get("YOCO_NVCC_EXTRA", ""))
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC] + (["-DYOCO_DEBUG_CHECKS"] if debug else []) + extra


def _compile(src, out_dir, debug):
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC, "-c", os.path.join(CSRC, src), "-o", obj] + _flags(debug)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose=False, debug=False):
    out_dir, lib = (DEBUG_DIR, DEBUG_LIB) if debug else (OUT_DIR, LIB)
    os.makedirs(out_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda src: _compile(src, out_dir, debug), SOURCES))
    if verbose:
        for _, err in results:
            if err:
                print(err)
    objs = [o for o, _ in results]
    cmd = [NVCC, "-shared", "-o", lib] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    subprocess.run(cmd, check=True)
    return lib


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, debug="--debug" in sys.argv))
