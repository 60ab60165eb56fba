"""GB300-native decode attention over a quantized, paged KV cache.

The compute path is a C-ABI CUDA library (``include/kvq.h``); ``kvq`` binds its
entry points for Python callers and ``synth`` draws seeded workloads."""
