"""CPU oracle for MXFP8 causal packed attention (test infrastructure only).

This package is the checker, not the product.  Only the tests, the smoke
entry point and the benchmark's CPU-baseline leg may import it; the CUDA
library never calls it and shares no code with it.

It is written from "FLAMIA: FLAsh MIcroscaling Attention for Fast and Causally
Safe Training on Blackwell" (arXiv 2611.03344) and holds two references:

* ``exact``  - exact fp64 softmax attention per document (Section 2,
  "FlashAttention" paragraph), forward and backward, no quantization.
* ``simulated`` - the same computation with every quantizer the method
  applies, simulated exactly: E4M3 codes with UE8M0 power-of-two scales
  (Section 2, "Microscaling floating-point formats"), document-local 32-token
  blocks (Sections 3.1 and 3.6.1), round-up exponents (Section 3.2), the fixed
  2^c probability multiplier with conditional rescale tau (Section 3.4 and
  Appendix B.1), D from the quantized dO (Section 3.3), 32x32 dS blocks
  (Section 3.3) and the 2^8 dV probability operand (Appendix B.1).

Parity status per function is stated in each module header.  Every function
in ``formats`` and ``blocks`` is pinned by tests against hand-worked values,
exhaustive enumeration or brute force; ``exact`` is pinned against textbook
softmax, a library attention routine and finite differences; ``simulated``
is pinned by reduction to ``exact`` with quantizers switched off, by the
saturation example of Appendix B.1, and by causality invariants.  The precise
rounding of P-hat and dS-hat codes near ties is *parity unpinned* (the GPU
rounds fp32 intermediates, the oracle rounds fp64 ones); it is covered by
tolerance only.
"""
from . import formats, blocks, exact, simulated  # noqa: F401
