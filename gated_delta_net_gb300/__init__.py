"""GB300-native speculative-tree verification through a Gated Delta Net layer.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA kernels
(``csrc/``, declared in ``include/gdn_tree.h``); ``binding`` marshals torch
tensors into it.  Importing this package does not load the library; the first
call does, and fails loudly if it was not built.
"""
__all__ = ["workloads", "binding"]
