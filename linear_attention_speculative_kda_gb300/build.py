"""Compile the CUDA library ``libkda.so`` in-tree for sm_103a.

Three translation units in one nvcc call, one ``-gencode`` (compute_103a /
sm_103a), the CUDA runtime linked statically so the library only needs the
driver at run time.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("kda_kernels.cu", "kda_conv.cu", "kda_blocks.cu")]
DEPENDS = SOURCES + [
    os.path.join(CSRC, "kda_device.cuh"),
    os.path.join(CSRC, "kda_async.cuh"),
    os.path.join(CSRC, "kda_align.cuh"),
    os.path.join(CSRC, "kda_tc.cuh"),
    os.path.join(ROOT, "include", "kda.h"),
]
LIBRARY = os.path.join(PKG, "libkda.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return os.path.join(cuda_home, "bin", "nvcc")


def _stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    built = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(src) > built for src in DEPENDS)


def compile_command(output: str, extra=(), sources=None) -> list[str]:
    return [
        nvcc_path(),
        *ARCH_FLAGS,
        "-O3",
        "-lineinfo",
        "-std=c++17",
        "-shared",
        "-Xcompiler",
        "-fPIC",
        "-cudart",
        "static",
        "-I",
        os.path.join(ROOT, "include"),
        *extra,
        "-o",
        output,
        *(SOURCES if sources is None else sources),
    ]


def build(force: bool = False, verbose: bool = False) -> str:
    """Build ``libkda.so`` if any source is newer than it; return its path."""
    if not force and not _stale():
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    extra = ["-Xptxas", "-v"] if verbose else []
    subprocess.run(compile_command(tmp, extra), check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


VARIANT_DIR = os.path.join(PKG, "_variants")


def build_variant(name: str, defines, force: bool = False) -> str:
    """Build a test variant of the library with extra preprocessor
    definitions, into _variants/libkda_<name>.so; never the product library.
    The tests use it for paths no input of the C ABI can reach (a wait that
    runs out)."""
    os.makedirs(VARIANT_DIR, exist_ok=True)
    out = os.path.join(VARIANT_DIR, f"libkda_{name}.so")
    if not force and os.path.exists(out) and not _stale_against(out):
        return out
    tmp = out + f".tmp{os.getpid()}"
    extra = [f"-D{d}" for d in defines]
    subprocess.run(compile_command(tmp, extra), check=True)
    os.replace(tmp, out)
    return out


def _stale_against(path: str) -> bool:
    built = os.path.getmtime(path)
    return any(os.path.getmtime(src) > built for src in DEPENDS)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
