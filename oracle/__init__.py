"""Plain fp64 CPU oracle for the quantized routed-expert MoE layer.

TEST INFRASTRUCTURE ONLY.  This package states, slowly and obviously, what the
GPU library computes, so that the CUDA path can be checked against it.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import it; the product path (the C-ABI library and its Python binding) never
does, and shares no code, header, table or helper with it.

Modules
-------
``oracle.quant``
    The packed 4-bit group-quantized weight format: quantize, dequantize, and the
    gate/up row interleave.  The pages name the EXL3 trellis codebook but do not
    define it (glm53-flash-offload README, "CPU tier" bullet), so the format is
    this library's own.
``oracle.moe``
    Router (sigmoid scores, top-k, renormalise), dispatch (histogram, stable
    permutation, active list), the SwiGLU expert FFN on dequantized weights, the
    shared expert, and the routing-weighted combine.

Every function cites the passage it follows.  All parts are pinned by tests
against closed forms, hand-derived fixtures, invariants and brute force; none
says "parity unpinned".
"""

from . import quant, moe  # noqa: F401
