"""GB300-native quantized MoE decode step: a C-ABI CUDA library and its binding.

Importing the package does not load the CUDA library; ``binding.load()`` does.
"""
