"""Sparse top-k routed MoE layer forward for NVIDIA B300 (sm_103a).

The hot path lives in hand-written CUDA kernels behind a C ABI (libmoe.so, declared in
include/moe.h).  `binding` marshals torch tensors into those calls; nothing on the path
runs on the host.
"""

__all__ = ["configs", "inputs"]
