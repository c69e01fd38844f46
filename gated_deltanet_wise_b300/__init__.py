"""B300-native frame-wise Gated DeltaNet forward pass.

The compute lives in the CUDA shared library ``libgdn_b300.so`` (C ABI declared
in ``include/gdn.h``); ``gated_deltanet_wise_b300.gdn`` is the thin ctypes
binding over it.  The library is loaded lazily on first use so that the input
generator in ``inputs`` can be imported on machines without the build.
"""

__all__ = ["gdn", "inputs"]
