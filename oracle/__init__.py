"""CPU oracle of the FastOCR decode-attention path (fp64 NumPy).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg. The product path (the CUDA library and its
binding) never imports, links or runs anything here, and this package shares
no code with it.

Modules:
  attention -- one layer: full, focal (score + top-k), sparse (gather) and
               R-SWA attention on one sequence.
  schedule  -- one decode step over all layers: warm-up profiling, focal set,
               Cross-Step Fixation Reuse (F_last).

Pins (tests/test_oracle_pins.py): every function is checked against something
other than itself -- PyTorch's fp64 scaled_dot_product_attention, closed
forms (constant keys, single-token sets, one-hot values), exhaustive search
over all k-subsets for the selection rule, and the invariants tau=1 => full
attention, R-SWA == full attention while T <= n, and total probability mass.
The end-task quality figure of the pages (98% accuracy) needs trained models
and is not part of this oracle: parity unpinned for that claim only.
"""
from . import attention, schedule  # noqa: F401
