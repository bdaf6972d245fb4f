"""Plain, slow CPU oracle of the paged KV cache hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code with the CUDA path (no kernels, headers, helpers or tables) and does
not import the ``paged_decode_attention_store_gb300`` package; the seeded
input generators are the only thing both sides consume, and they are passed
in as plain arrays.

Parts
-----
``pagetable``      block table, LIFO free list, reference counts, fork, lazy
                   copy-on-write and window trim ("A Paged KV Cache and
                   Sliding-Window Attention", section "The model"), plus the
                   position translation of "PagedAttention block allocator",
                   section "Sequence block table".
``raw_locations``  the raw token-location page table of the mini-sglang code
                   series, part 4 (allocation counted in pages, recorded in
                   tokens, one scatter write, dummy row and dummy page).
``attention``      dense masked softmax attention over the rows gathered
                   through a table, in float64 ("Week 3 Day 3: Paged KV
                   Cache", section "Correctness Checkpoint: Gather Pages for
                   Dense Attention").

Every function is pinned by ``tests/test_oracle_*.py`` to values the pages
print, closed forms, invariants or library routines; none is "parity
unpinned".
"""

from . import pagetable, raw_locations, attention, decode  # noqa: F401
