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


def _stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    built = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(src) > built for src in SOURCES)


def build(force: bool = False) -> str:
    """Compile the oracle if needed and return the library path."""
    if not force and not _stale():
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = [
        os.environ.get("CC", "gcc"),
        "-O2",
        "-std=c11",
        "-ffp-contract=off",
        "-fno-fast-math",
        "-fPIC",
        "-shared",
        "-o",
        tmp,
        *SOURCES,
        "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
