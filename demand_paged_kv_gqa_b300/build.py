"""Build libgrowpage.so in-tree with nvcc for sm_103a (B300).

Usage: python -m demand_paged_kv_gqa_b300.build  (or call build()).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libgrowpage.so")
SOURCES = ["gp_host.cu", "gp_attn.cu", "gp_attn_mma.cu", "gp_ceiling.cu", "gp_step.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_cmd(out=LIB, extra=()):
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    # -fno-builtin-*: the host RoPE table must come from the C library's own
    # pow/cos/sin calls (no compiler substitution such as sincos fusion).
    return [nvcc, "-std=c++17", "-O3", ARCH, "-lineinfo", "--shared",
            "-Xcompiler", "-fPIC,-fno-builtin-sin,-fno-builtin-cos,-fno-builtin-sincos,-fno-builtin-pow",
            "-I", INCLUDE, "-I", CSRC, "-o", out,
            *[os.path.join(CSRC, s) for s in SOURCES], "-lcudart", *extra]


def build(verbose=False, extra=()):
    cmd = nvcc_cmd(extra=extra)
    if verbose:
        print(" ".join(cmd))
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr)
    return LIB


if __name__ == "__main__":
    build(verbose=True, extra=sys.argv[1:])
