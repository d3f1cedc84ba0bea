"""GB300-native exact softmax attention (FlashAttention-style) behind a C ABI.

The compute path is libfa.so (hand-written sm_103a kernels, see include/fa.h);
``online_softmax_09_gb300.fa`` is its ctypes binding. Importing this package loads
nothing: the library is opened on first use and its absence raises.
"""

__all__ = ["fa", "inputs", "build"]
