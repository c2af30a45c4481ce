"""Build libmlaq.so in-tree with nvcc for sm_103a (no CMake, one nvcc call)."""

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ["mlaq_api.cu", "mlaq_writer.cu", "mlaq_decode.cu"]
LIB = os.path.join(HERE, "libmlaq.so")


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile the CUDA sources into bit_mla_kv_gb300/libmlaq.so; returns its path.

    Extra nvcc flags (experiments) may be given in MLAQ_NVCC_FLAGS."""
    srcs = [os.path.join(HERE, "csrc", s) for s in SOURCES]
    deps = srcs + [os.path.join(HERE, "csrc", "mlaq_internal.cuh"), os.path.join(HERE, "csrc", "mlaq_decode_tc.cuh"),
                   os.path.join(HERE, "..", "include", "mlaq.h")]
    extra = os.environ.get("MLAQ_NVCC_FLAGS", "").split()
    if extra:
        force = True
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(d) for d in deps)
        if os.path.getmtime(LIB) >= newest:
            return LIB
    cmd = [nvcc_path(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-o", LIB + ".tmp"] + extra + srcs
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + proc.stdout + proc.stderr)
    if verbose:
        print(proc.stdout + proc.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, force=True))
