"""GB300-native block-cached decoding kernels (Fast-dLLM hot path).

Importing the package loads nothing native; `block_cached_decoding_gb300.fdllm`
loads the CUDA library and raises if it is missing.
"""
