"""Build libpagedkv.so on demand for the tests (nvcc cross-compiles without a GPU)."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_done = False


def ensure_built():
    global _done
    if not _done:
        from paged_decode_attention_store_gb300 import build

        build.build()
        _done = True
    from paged_decode_attention_store_gb300 import binding

    return binding
