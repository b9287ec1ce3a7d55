"""TurboQuant-style KV-cache compression and compressed-cache decode attention for GB300.

The compute path is the native library ``libtq.so`` (hand-written CUDA for
sm_103a behind a C ABI, declared in ``include/tq.h``); ``tq`` is its thin
ctypes binding and ``workloads`` holds the seeded synthetic inputs.  Import
``kv_cache_quantization_turbo_gb300.tq`` to load the library.
"""
