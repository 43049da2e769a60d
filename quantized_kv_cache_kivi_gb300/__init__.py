"""GB300-native decode attention over a KIVI / WindowQuant quantized KV cache.

Importing the package loads nothing native; the CUDA library is loaded on the
first call of the binding in ``kvq`` (and fails loudly when it is missing).
"""
