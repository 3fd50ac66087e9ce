"""GB300-native verify round of lossless speculative decoding.

The compute lives in ``libspecverify.so`` (hand-written CUDA for sm_103a behind
the C ABI in ``include/specverify.h``); ``binding`` is its thin ctypes layer
and ``build`` compiles it in-tree.  Importing this package loads nothing; call
``binding.load()`` to open the library.
"""
