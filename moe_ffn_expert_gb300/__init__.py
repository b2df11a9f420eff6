"""Fused MoE-FFN forward and backward for one GB300 GPU (sm_103a).

The layer runs in libmm.so (hand-written CUDA: routing, dispatch, tcgen05 grouped GEMMs with
fused SwiGLU / SwiGLU-backward epilogues, fixed-order combine) behind the C ABI in
include/mm.h. `_abi` is its ctypes binding; `torch_api` adds the PyTorch call
`hyper_mega_moe` and the workspace helper. Importing this package does not load the library;
the first call does, and fails loudly if it has not been built.
"""
from . import _abi  # noqa: F401

__all__ = ["_abi"]
