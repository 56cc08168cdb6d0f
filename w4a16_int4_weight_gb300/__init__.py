"""GB300-native W4A16 int4-weight linear layer.

``C[M,N] = A[M,K] . dequant(W)^T`` with a group-quantised 4-bit weight, computed
by hand-written sm_103a CUDA kernels behind the C ABI in ``include/w4a16.h``.

Importing the package loads nothing; ``w4a16_int4_weight_gb300.binding`` loads
``libw4a16.so`` (built by ``w4a16_int4_weight_gb300.build``) and raises if it is
missing.
"""

__all__ = ["binding", "build", "inputs"]
