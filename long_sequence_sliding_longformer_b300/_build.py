"""Builds the CUDA library liblf_attn.so in-tree for sm_103a (B300) with nvcc."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC_DIR = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "liblf_attn.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include", "lf_attn.h")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def _sources():
    return [os.path.join(SRC_DIR, f) for f in sorted(os.listdir(SRC_DIR))
            if f.endswith((".cu", ".cuh"))] + [INCLUDE]


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile csrc/lf_attn.cu (one translation unit) into liblf_attn.so."""
    newest = max(os.path.getmtime(p) for p in _sources())
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-o", tmp, os.path.join(SRC_DIR, "lf_attn.cu")]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
