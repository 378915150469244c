"""GB300-native linear layers over packed trellis-coded (QTIP 1MAD) weights.

The compute path is the CUDA library ``libtrellis.so`` (hand-written sm_103a
kernels behind a C ABI declared in ``include/trellis.h``); ``binding`` is its
thin ctypes layer.  PyTorch is used only for device memory and streams.
"""
__all__ = ["inputs"]
