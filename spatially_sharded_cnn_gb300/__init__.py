"""Width-sharded (halo-exchange) Conv2d forward and backward for GB300 (sm_103a).

The compute path is the C-ABI library built from ``csrc/`` (hand-written CUDA);
``spatially_sharded_cnn_gb300.hc`` is its thin ctypes binding and raises at
import when the library has not been built.  ``synth`` holds the seeded input
generators.
"""
__all__ = ["hc", "synth"]
