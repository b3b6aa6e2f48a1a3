"""GB300-native single-GPU MoE layer (router, deterministic dispatch,
tcgen05 grouped-GEMM SwiGLU experts, fixed-order combine, backward, forward
MegaKernel) behind a C ABI.  ``moe`` is the ctypes binding; importing this
package does not load the CUDA library."""
from .configs import MoEConfig, ALL, BY_NAME  # noqa: F401
