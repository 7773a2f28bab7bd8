"""fp64 CPU oracle for the paged-KV decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
the oracle imports nothing from the product package: the two share no code.

Contents
  * ``core``       -- ctypes wrapper of ``pa_oracle.c`` (cache write, block
                      copy, decode attention, E4M3 encode/decode), built with
                      gcc on first use.
  * ``pool_model`` -- a pure-Python model of the block pool and the per-
                      sequence block tables (free queue, ref counts, fork,
                      copy-on-write, slot mapping).
  * ``accounting`` -- the KV-size closed form and the utilisation estimator.

Parity status of each function is stated in its docstring; every function
here is pinned by a ``-m "not gpu"`` test against values or identities the
source pages fix (see tests/test_oracle_pins.py and tests/test_pool.py).
"""
