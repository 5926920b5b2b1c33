"""CPU oracle for the mega-kernelised decode step.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library
and its Python binding) never imports, links or executes anything here, and
this package imports nothing from the product.

Sources (cited by title and section throughout):
  * "MPK: A Compiler and Runtime for Mega-Kernelizing Tensor Programs"
    (paper summary page) -- called "MPK summary" below;
  * "Compiling LLMs into a MegaKernel: A path to low-latency inference"
    (the author's Hacker News comments) -- called "MegaKernel HN comments".

Modules:
  * ``numerics`` -- the decode step as plain NumPy: fp32 math on bf16
    values, rounding to bf16 (round-to-nearest-even) at tensor boundaries;
  * ``tgraph``   -- the reference tGraph builder: decomposition, overlap
    dependencies, event fusion (Defs 4.1/4.2), normalisation, BFS
    linearisation, AOT worker assignment.

Parity status: every function is pinned by tests under ``tests/`` against
library routines, closed forms, invariants or hand-worked fixtures.  The
pages print no numeric worked example of a whole decode step, so the
end-to-end model outputs are pinned only through those per-step checks and
the decode-vs-full-sequence consistency check.
"""
