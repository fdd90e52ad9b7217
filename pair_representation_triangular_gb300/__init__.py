"""Starting-node triangular self-attention over a pair representation, forward
pass, as a GB300-native (sm_103a) CUDA library with a thin Python binding.

``binding`` holds the ctypes binding of include/tri_attn.h (same names as the C
entry points) and ``TriangularAttention``; ``workloads`` draws seeded synthetic
inputs; ``build`` compiles the library in-tree.
"""
__all__ = ["binding", "workloads", "build"]
