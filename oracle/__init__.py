"""FP64 CPU oracle for the BF16-activation x FP4-weight GEMM.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and
its Python binding) imports, calls or links anything in this package; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code, tables
or constants with ``fp4_weight_only_gb300/``.

What it computes (sources are the four web pages on the method):

* ``formats``  -- the number formats: E2M1 (FP4), E4M3FN, E8M0, BF16.
* ``quantize`` -- NVFP4 (16-element E4M3 block scale + FP32 global scale) and
  MXFP4 (32-element E8M0 block scale) quantizers and the two-per-byte packing.
* ``gemm``     -- exact dequantisation ``Wq = code * block_scale`` and the
  reference product ``C = g * A . Wq^T`` in float64.

Every function is pinned by ``tests/test_oracle_*.py`` (``-m "not gpu"``)
against closed forms, library casts, invariants and brute force.  No part of
the oracle is "parity unpinned".
"""

from . import formats, quantize, gemm  # noqa: F401
