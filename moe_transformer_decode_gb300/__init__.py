"""GB300-native single-kernel decode step for parallel-layer MoE transformers.

The compute path is libmk.so (CUDA for sm_103a) behind the C ABI in include/mk.h; the
Python names below only marshal arguments into that ABI (see binding.py).
"""
