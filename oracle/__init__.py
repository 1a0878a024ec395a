"""CPU oracle for the fused operators: plain, slow, unfused, float64.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
cpu_baseline / reference arm of bench.py may import or run anything here.
The product path (fusion_add_rmsnorm_gb300 and its CUDA library) never
imports it, and this package imports nothing from the product path: the two
share no code.  The only code both sides use is the seeded input generator
module `workloads`, which holds none of the operators' arithmetic.

Modules:
  formats -- bfloat16 and OCP FP8 E4M3 codecs written from the bit layouts
  ops     -- one function per unfused operator (residual add, RMSNorm, AdaRMSNorm
             modulation, static FP8 quantisation, rotate_half / 3D RoPE, packed
             QKV split, Linear, GELU-tanh, BatchNorm, BN folding, direct conv)
  chains  -- the operator chains each fused kernel replaces, bits in, bits out

Every function is pinned by tests/test_oracle_*.py to facts that do not come
from the oracle itself: closed forms, hand-derived worked examples in
tests/golden/, library routines on special cases, invariants and brute force.
"""
from . import formats, ops, chains  # noqa: F401
