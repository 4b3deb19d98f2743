"""GB300-native canonical Huffman coding of ML tensor bytes.

The compute lives in ``libhuff.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/huff.h``).  ``_lib`` is the thin ctypes binding with
the same function names; ``workloads`` draws the seeded synthetic inputs.
The binding is imported lazily so that ``workloads`` can be used without the
CUDA library.
"""
__all__ = ["workloads"]
