"""Build the CPU oracle's shared library with gcc (test infrastructure only).

The oracle is plain C compiled with strict IEEE double arithmetic
(``-ffp-contract=off``, no fast-math), so that it gives the same results on
x86-64 and on AArch64 hosts.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = [os.path.join(HERE, "kda_window.c")]
LIBRARY = os.path.join(HERE, "libkda_oracle.so")
# the same source built with float arithmetic: timed by the benchmark's CPU
# baseline beside the oracle, never used by a test
LIBRARY_FP32 = os.path.join(HERE, "libkda_oracle_fp32.so")


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    built = os.path.getmtime(path)
    return any(os.path.getmtime(src) > built for src in SOURCES)


def _compile(path: str, defines=()) -> None:
    tmp = path + f".tmp{os.getpid()}"
    cmd = [
        os.environ.get("CC", "gcc"),
        "-O2",
        "-std=c11",
        "-ffp-contract=off",
        "-fno-fast-math",
        "-fPIC",
        "-shared",
        *defines,
        "-o",
        tmp,
        *SOURCES,
        "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)


def build(force: bool = False) -> str:
    """Compile the oracle (and its float build) if needed; return the
    oracle's library path."""
    if force or _stale(LIBRARY):
        _compile(LIBRARY)
    if force or _stale(LIBRARY_FP32):
        _compile(LIBRARY_FP32, ["-DKDA_ORACLE_FP32"])
    return LIBRARY


def library(arithmetic: str = "fp64") -> str:
    """Path of the built library for 'fp64' (the oracle) or 'fp32'."""
    build()
    return LIBRARY if arithmetic == "fp64" else LIBRARY_FP32


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
