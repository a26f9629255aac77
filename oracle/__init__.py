"""CPU oracle for the SageAttention3-style quantized attention forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) imports, calls or links this package; only the tests,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.  It shares no code with the CUDA path.

Contents (each function cites the passage it follows; page names are those of
the source pages):

* ``formats``   -- e2m1 (FP4) and e4m3 (FP8) codecs.  Page "GPU kernel porting
  with AI agents", section "Sage Attention 3": FP4 e2m1 has 15 representable
  values, NVFP4 groups are 1x16 with FP8 e4m3 scale factors.
* ``quant``     -- smooth-K mean and 1x16 NVFP4 group quantisation of Q, K, V
  (same section; smooth-K from page "kernel overview", SageAttention
  technique chain).
* ``layout``    -- the byte layout the C ABI documents for packed codes and
  scale factors (a statement of the interface, written independently of the
  CUDA sources).
* ``attention`` -- exact FP64 softmax attention and the tile-by-tile emulation
  of the SA3 scheme (online softmax from page "FlashAttention kernels" section
  0/1; two-level P quantisation from "Sage Attention 3").

All arithmetic is NumPy, in FP64 except where the scheme fixes FP32 (the
quantiser steps), which are done in float32 with IEEE round-to-nearest-even.
Parity unpinned: nothing; every function has at least one pin in
``tests/test_oracle_*.py`` (closed forms, invariants, hand-worked examples,
an independent torch FP8 cast, brute force on tiny inputs).
"""

from . import formats, quant, layout, attention  # noqa: F401
