"""GB300-native decode step of Multi-head Latent Attention (forward_absorb path).

``libmla_decode.so`` (C ABI, ``include/mla_decode.h``) holds the sm_103a
kernels; ``binding`` is its ctypes binding; ``inputs`` draws the seeded
synthetic workloads; ``build`` compiles the library in-tree.
"""
__all__ = ["binding", "build", "inputs"]
