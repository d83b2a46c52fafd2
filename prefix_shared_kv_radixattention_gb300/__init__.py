"""Prefix-shared KV attention over a token-slot pool, for GB300 (sm_103a).

The compute path lives in a C-ABI shared library (``include/rx.h``) built from
``csrc/``; ``prefix_shared_kv_radixattention_gb300.binding`` is its thin ctypes
layer and loads the library on import.  ``inputs`` only draws seeded inputs
and loads nothing.
"""
