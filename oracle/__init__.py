"""fp64 CPU oracle for the sparse-attention hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, step-by-step
restatement of what the pages define, written in numpy float64.  Only the
test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import it.  The product path (the CUDA library and its
Python binding) never imports, calls or links anything here, and nothing here
imports the product path.

Modules:
  hip   -- InfiniteHiP pruning stages (candidate range, chunking, SelectRep,
           chunk score, top-K, index assembly) and split-free sparse decode
           attention over sink + selected + window keys.
  vs    -- MInference vertical-slash estimate, top-k, conversion to the tiled
           block/column format, and sparse causal prefill attention.
  patterns -- MInference A-shape (static initial blocks + diagonal band) and
           Block-Sparse (mean-pooled block attention, top-k_b blocks) lists.
  numerics -- exact widening of the stored bit patterns to float64.

Pinning status (what each function is checked against) is listed in the
module docstrings; the selection heuristic's tie readings are pinned only by
the written readings of the pages (see the "parity unpinned" notes).
"""
from . import hip, numerics, patterns, vs  # noqa: F401
