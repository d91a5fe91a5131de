"""CPU check that the C ABI is usable from plain C.

A C99 program (strict, warnings as errors) includes ``include/kda.h``, takes
the address of every entry point the header declares, links against the
in-tree ``libkda.so`` and calls the entry points that never launch a kernel:
the records-size helpers, the status names, the ABI version, and a call
with no rows.  No GPU is touched.
"""

import os
import re
import shutil
import subprocess

import pytest

from linear_attention_speculative_kda_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>

#include "kda.h"

typedef void (*any_fn)(void);

int main(void) {
    /* every entry point the header declares, by address */
    any_fn fns[] = {%(fns)s};
    size_t i;
    for (i = 0; i < sizeof fns / sizeof fns[0]; ++i)
        if (fns[i] == NULL) return 10;
    if (kda_records_bytes(16, 4, 1024) != (size_t)1025 * 16 * 4 * 392 * 2) return 1;
    if (kda_correction_records_bytes(16, 4, 1024) != (size_t)1025 * 16 * 4 * 1024) return 2;
    if (kda_records_bytes(4, 9, 4) != 0) return 3;
    if (strcmp(kda_status_string(KDA_ERR_INVALID_ARG), "KDA_ERR_INVALID_ARG") != 0) return 4;
    if (kda_abi_version() != 4) return 5;
    /* no rows: nothing is inspected or launched */
    if (kda_record_state_blocks(NULL, NULL, NULL, 0, NULL, NULL, 0, NULL, NULL) != KDA_OK)
        return 6;
    if (kda_record_state_blocks(NULL, NULL, NULL, -1, NULL, NULL, 0, NULL, NULL) !=
        KDA_ERR_INVALID_ARG)
        return 7;
    printf("ok %%u\n", (unsigned)(sizeof fns / sizeof fns[0]));
    return 0;
}
"""


def _declared():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_compiles_and_links_as_c99(tmp_path):
    lib = kbuild.build()
    names = _declared()
    src = tmp_path / "use_kda.c"
    src.write_text(PROGRAM % {"fns": ", ".join(f"(any_fn){n}" for n in names)})
    exe = tmp_path / "use_kda"
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lkda",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == f"ok {len(names)}"
