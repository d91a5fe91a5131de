"""CPU oracle of KDA speculative verify/commit -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product library never does.
"""
