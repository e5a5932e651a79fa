"""Build the CUDA library libdecode_attn.so in-tree for GB300 (sm_103a).

One translation unit (decode_attn.cu, which includes multi_attn.cuh), nvcc, static CUDA runtime; the driver API entry used
for tensor maps is resolved at run time, so the library loads on a machine
without a GPU (for the ABI checks) and needs no libcuda at link time.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "decode_attn.cu")
HDR = os.path.join(ROOT, "include", "decode_attn.h")
LIB = os.path.join(HERE, "libdecode_attn.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, extra_flags=(), out: str = LIB, verbose: bool = False) -> str:
    """Compile the library unless it is newer than its sources."""
    csrc = os.path.dirname(SRC)
    deps = [os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith((".cu", ".cuh"))] + [HDR]
    newest = max(os.path.getmtime(f) for f in deps)
    if not force and not extra_flags and os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include"),
           *extra_flags, SRC, "-o", tmp]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, extra_flags=sys.argv[1:], verbose=True))
