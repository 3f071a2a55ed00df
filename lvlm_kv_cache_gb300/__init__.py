"""GB300-native AirCache: one-shot post-prefill visual KV-cache compression.

The compute path is the CUDA library ``libaircache.so`` built from ``csrc/``
(C ABI declared in ``include/aircache.h``); ``aircache`` is its thin ctypes
binding and ``workloads`` draws seeded synthetic inputs.  Submodules are
imported explicitly so that loading the package does not load the library.
"""
