"""NVFP4 / MXFP8 linear-layer kernels for one GB300 (sm_103a).

``fp4q`` is the ctypes binding over the C-ABI library ``libfp4q.so`` (import it
explicitly: it fails loudly when the library has not been built); ``inputs``
holds the seeded synthetic input generators; ``layer`` composes the entry points
into the forward and backward pass of the NVFP4 linear layer and MLP block.
"""
__all__ = ["fp4q", "inputs", "layer"]
