"""Batch-invariant mHC pre "H Aggregate" for GB300 (sm_103a).

``out[t,h] = bf16((pre0*r0 + pre1*r1) + (pre2*r2 + pre3*r3))`` over a BF16
residual ``[T,4,H]`` and FP32 ``pre`` ``[T,4]``, and its fused backward, as
hand-written CUDA behind a C ABI (``include/mhc_h_aggregate.h``).

Importing the package loads nothing; the CUDA library is loaded on first use
by :mod:`invariant_mhc_aggregate_gb300.binding`, which raises if it has not
been built (``invariant_mhc_aggregate_gb300._build.build()``).
"""

__all__ = ["autograd", "binding", "inputs", "sharding"]
