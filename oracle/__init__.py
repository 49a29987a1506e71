"""Oracle for the fused large-vocabulary LM cross-entropy: TEST INFRASTRUCTURE.

Plain, slow and obviously correct CPU implementations (fp64) of what the CUDA
library computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never loads it.

* :mod:`oracle.ce`   -- cross-entropy forward + backward (C, fp64, threads).
* :mod:`oracle.flce` -- fused linear cross-entropy, as fp64 matmuls composed
  with the cross-entropy oracle.

Parity pins: every function here is pinned by ``tests/test_oracle.py`` and
``tests/test_oracle_flce.py`` to closed forms, invariants, finite differences,
brute force and library special cases.  No function is "parity unpinned".
"""
