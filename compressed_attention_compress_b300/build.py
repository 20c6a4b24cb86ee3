"""Build libhsa.so in-tree with nvcc for sm_103a (no GPU needed to compile)."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libhsa.so")
SOURCES = ["hsa_api.cu", "compress.cu", "index_topk.cu", "index_fused.cu", "attn.cu", "attn_decode_cluster.cu", "attn_prefill_tc.cu", "index_prefill_tc.cu", "cp_merge.cu", "v4_extras.cu", "attn_gather_tc.cu", "attn_decode_tc.cu", "attn_decode_dense_tc.cu", "decode_fused.cu"]
HEADERS = ["common.cuh", "internal.h", "block_scan.cuh", "tc_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "hsa.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr", "-rdc=true",
           "-I", os.path.join(ROOT, "include"), "-o", LIB + ".tmp"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    cmd += [os.path.join(CSRC, f) for f in SOURCES]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
