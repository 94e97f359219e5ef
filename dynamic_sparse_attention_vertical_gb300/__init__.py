"""GB300-native dynamic sparse prefill attention (vertical-slash, block-sparse, A-shape).

The compute lives in hand-written CUDA kernels for sm_103a behind the C ABI in
``include/mi.h`` (``libmi.so``).  ``binding`` marshals torch tensors into that
ABI; it loads the library on first use and raises if it is missing.
"""
__all__ = ["binding", "inputs", "search"]
