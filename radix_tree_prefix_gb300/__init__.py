"""GB300-native RadixAttention hot path: a host radix cache over a
token-granular KV pool plus sm_103a CUDA kernels, behind a C ABI (librx.so).

Importing the package loads nothing; ``radix_tree_prefix_gb300.rx`` loads the
native library and raises if it has not been built.
"""
