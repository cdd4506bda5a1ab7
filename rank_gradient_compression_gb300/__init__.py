"""GB300-native PowerSGD gradient compression with error feedback (libpsgd.so + binding).

Import ``rank_gradient_compression_gb300.psgd`` for the ctypes binding; it raises if the
CUDA library has not been built (``python -m rank_gradient_compression_gb300.build``).
"""
__all__ = ["psgd", "build"]
