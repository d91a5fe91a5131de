"""GB300-native KDA speculative verify and commit (RecoverSSM).

The compute path is a C-ABI CUDA library (``libkda.so``, sm_103a) whose entry
points are declared in ``include/kda.h``; :mod:`.api` is a thin ctypes binding
with the same names.  Importing the package does not load the library; the
first call does, and fails loudly if it has not been built.
"""

from .api import (  # noqa: F401
    KDAError,
    kda_commit,
    kda_flush,
    kda_records_bytes,
    kda_verify,
    library_path,
)
