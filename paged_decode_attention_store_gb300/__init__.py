"""GB300-native paged decode attention and store_cache.

The compute path is the C-ABI shared library ``libpagedkv.so`` built from
``csrc/`` (hand-written CUDA for sm_103a plus the host-side page-table
bookkeeping in C++). :mod:`.binding` loads it and exposes the same entry
points to Python; it fails loudly when the library is missing.
:mod:`.workloads` holds the seeded synthetic inputs.
"""

__all__ = ["binding", "workloads"]
