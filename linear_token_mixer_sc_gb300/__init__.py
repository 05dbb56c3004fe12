"""GB300-native Interdomain Attention token mixer (prefill + recurrent decode).

The compute path is the CUDA library ``libida.so`` (built from ``csrc/``);
``binding`` marshals torch tensors into its C ABI.  Importing this package
loads nothing; the library is loaded on first use and a missing library is
an error, never a fallback.
"""
__all__ = ["binding", "configs", "inputs"]
