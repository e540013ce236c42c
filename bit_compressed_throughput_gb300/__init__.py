"""GB300-native INT4 group-compressed OPT layer engine.

The compute path is ``libfg.so``: hand-written sm_103a CUDA kernels behind a C ABI
(``include/fg.h``).  ``bit_compressed_throughput_gb300.fg`` is its thin ctypes binding;
importing it loads the library and fails loudly when it has not been built.
``accounting`` holds host-side byte and flop counts.  Nothing here falls back to a CPU
implementation.
"""
__all__ = ["accounting"]
