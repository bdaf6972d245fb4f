"""Block-table bookkeeping oracle (test infrastructure only; see ``oracle``).

Restates, in plain Python, the page table of "A Paged KV Cache and
Sliding-Window Attention" (silicon_compiler_from_scratch, chapter 15,
section "The model"):

* the pool has ``n_pages`` physical pages of ``page`` token rows each;
* the free list is a stack: the page at the END of the list is handed out
  next, and a page whose last owner lets go is pushed back on the end. The
  chapter starts it as ``n-1 … 0`` so that page 0 goes out first; a seeded
  shuffle may be given instead;
* a request owns a block table (its live physical pages in logical order),
  a length (rows stored) and a ``dropped`` count (front pages released by
  the window). Logical page ``i`` lives at ``table[i - dropped]``;
* appending row ``i`` takes a fresh page when ``i % page == 0``; otherwise,
  if the tail page is shared (reference count > 1), it first copies the
  whole tail page into a fresh page, lets go of the shared one and writes
  into the copy (lazy copy-on-write);
* ``trim(keep_from)`` releases front pages whose rows all lie below
  ``keep_from``: page ``dropped`` goes while ``(dropped + 1) * page <=
  keep_from``;
* with attention sinks (the chapter's exercise "Attention sinks": the first
  ``S`` rows stay in every context), ``trim(keep_from, sink_rows=S)`` keeps
  the first ``ceil(S / page)`` pages and releases the ones after them the
  same way: page ``sp + dropped`` goes while ``(sp + dropped + 1) * page <=
  keep_from``. Logical page ``i`` then lives at ``table[i]`` for ``i < sp``
  and at ``table[i - dropped]`` from ``sp + dropped`` on (the chapter gives
  no bookkeeping for sinks; this is the plain reading that releases exactly
  the pages no later step reads);
* ``fork`` copies table, length and dropped count and adds one reference to
  every page; ``release`` lets go of every page;
* ``rewind(n)`` ("Week 3 Day 3: Paged KV Cache", tiny-llm: drop the newest
  ``n`` logical tokens, free the whole pages no longer needed and shorten
  the valid length of the last page that remains) lets go of the pages past
  ``ceil((length - n) / page)``. The page is silent on the order in which
  freed pages return; they are pushed tail first, so that the stack hands
  them back in logical order and re-appending the same tokens rebuilds the
  same table. Rows that a later step may read must stay: the new length may
  not reach below the released front (the window's or the sinks' holes).

Exhaustion raises :class:`OutOfPages` before any state changes, so a failed
append leaves the request untouched (chapter 15, section "Tests", item 2).

Position translation follows "PagedAttention block allocator", section
"Sequence block table": position ``t`` lives in logical page ``t // P`` at
offset ``t % P``; outside ``[0, length)`` it is an error.

The device-facing view used by the GPU path is :meth:`PageTable.block_row`:
a row indexed by ABSOLUTE logical page, with ``-1`` for pages the window has
released (the "hole at the front of the table" of chapter 15, Figure 15.1;
behind the sink pages when there are sinks).
"""

from __future__ import annotations


class OutOfPages(Exception):
    """No free physical page is left."""


class PageTable:
    def __init__(self, n_pages: int, page: int = 4, free_order=None):
        if n_pages <= 0 or page <= 0:
            raise ValueError("n_pages and page must be positive")
        self.page = page
        self.n_pages = n_pages
        # The free list is a stack whose top is the end of the list.
        if free_order is None:
            self.free = list(range(n_pages - 1, -1, -1))
        else:
            self.free = [int(p) for p in free_order]
            if sorted(self.free) != list(range(n_pages)):
                raise ValueError("free_order must be a permutation of 0..n_pages-1")
        self.ref = [0] * n_pages
        # Row storage: pool[page][offset]; rows are opaque objects.
        self.pool = [[None] * page for _ in range(n_pages)]
        self.table: dict = {}
        self.length: dict = {}
        self.dropped: dict = {}
        self.sinks: dict = {}  # sink pages kept in front of the released ones

    # -- pool ---------------------------------------------------------------
    def _alloc(self) -> int:
        if not self.free:
            raise OutOfPages("no free page")
        p = self.free.pop()
        self.ref[p] = 1
        return p

    def _unref(self, p: int) -> None:
        self.ref[p] -= 1
        if self.ref[p] == 0:
            self.free.append(p)

    def used(self) -> int:
        """Pages currently owned by at least one request."""
        return self.n_pages - len(self.free)

    # -- requests -------------------------------------------------------------
    def new(self, rid) -> None:
        self.table[rid] = []
        self.length[rid] = 0
        self.dropped[rid] = 0
        self.sinks[rid] = 0

    def append(self, rid, row=None) -> dict:
        """Store one row at the end of request ``rid``.

        Returns where it went: ``slot`` (= physical page * P + offset, the
        flat token location), the logical page, the fresh page taken (or
        None) and the copy-on-write pair ``(shared_page, private_copy)`` (or
        None).
        """
        i = self.length[rid]
        off = i % self.page
        t = self.table[rid]
        new_page = None
        cow = None
        if off == 0:
            new_page = self._alloc()
            t.append(new_page)
        else:
            shared = t[-1]
            if self.ref[shared] > 1:
                q = self._alloc()
                self.pool[q] = list(self.pool[shared])  # whole-page copy
                self._unref(shared)
                t[-1] = q
                cow = (shared, q)
        phys = t[-1]
        self.pool[phys][off] = row
        self.length[rid] = i + 1
        return {
            "slot": phys * self.page + off,
            "page": phys,
            "offset": off,
            "logical_page": self.dropped[rid] + len(t) - 1,
            "new_page": new_page,
            "cow": cow,
        }

    def translate(self, rid, pos: int):
        """(physical page, offset) of logical position ``pos``."""
        if pos < 0 or pos >= self.length[rid]:
            raise IndexError(f"position {pos} outside [0, {self.length[rid]})")
        logical = pos // self.page
        sp, d = self.sinks[rid], self.dropped[rid]
        if logical < sp:
            return self.table[rid][logical], pos % self.page
        if logical < sp + d:
            raise IndexError(f"position {pos} lies in a released page")
        return self.table[rid][logical - d], pos % self.page

    def slot(self, rid, pos: int) -> int:
        """Flat token location ``page * P + offset`` of logical position ``pos``."""
        phys, off = self.translate(rid, pos)
        return phys * self.page + off

    def rows(self, rid, lo: int, hi: int) -> list:
        """Rows ``lo <= i < hi`` read back through the block table."""
        out = []
        for i in range(lo, hi):
            phys, off = self.translate(rid, i)
            out.append(self.pool[phys][off])
        return out

    def trim(self, rid, keep_from: int, sink_rows: int = 0) -> list:
        """Release the front pages that hold only rows below ``keep_from``,
        except the first ``ceil(sink_rows / page)`` pages.

        Returns the absolute logical indices of the released pages (they
        become ``-1`` holes in :meth:`block_row`).
        """
        sp = -(-sink_rows // self.page)
        if self.dropped[rid] > 0 and sp != self.sinks[rid]:
            raise ValueError("the sink pages of a request cannot change once pages are released")
        self.sinks[rid] = sp
        t = self.table[rid]
        released = []
        while len(t) > sp and (sp + self.dropped[rid] + 1) * self.page <= keep_from:
            self._unref(t.pop(sp))
            released.append(sp + self.dropped[rid])
            self.dropped[rid] += 1
        return released

    def rewind(self, rid, n: int) -> list:
        """Drop the newest ``n`` tokens; returns the absolute logical indices
        of the pages let go (tail first)."""
        L = self.length[rid]
        if n < 0 or n > L:
            raise ValueError(f"cannot rewind {n} of {L} tokens")
        keep_len = L - n
        sp, d = self.sinks[rid], self.dropped[rid]
        if d > 0 and keep_len < (sp + d) * self.page:
            raise ValueError("rewind would reach into released pages")
        keep_pages = -(-keep_len // self.page)  # absolute logical pages that keep rows
        t = self.table[rid]
        gone = []
        while t and d + len(t) > keep_pages and (d == 0 or len(t) > sp):
            logical = d + len(t) - 1
            self._unref(t.pop())
            gone.append(logical)
        self.length[rid] = keep_len
        return gone

    def fork(self, src, dst) -> None:
        self.table[dst] = list(self.table[src])
        self.length[dst] = self.length[src]
        self.dropped[dst] = self.dropped[src]
        self.sinks[dst] = self.sinks[src]
        for p in self.table[dst]:
            self.ref[p] += 1

    def release(self, rid) -> None:
        for p in self.table.pop(rid):
            self._unref(p)
        del self.length[rid]
        del self.dropped[rid]
        del self.sinks[rid]

    # -- device-facing views --------------------------------------------------
    def block_row(self, rid) -> list:
        """Block-table row indexed by absolute logical page, ``-1`` for holes.

        Covers logical pages ``0 .. dropped + len(table) - 1``: everything a
        decode step of this request can address.
        """
        t, sp = self.table[rid], self.sinks[rid]
        return list(t[:sp]) + [-1] * self.dropped[rid] + list(t[sp:])

    def raw_row(self, rid) -> list:
        """The same row expanded to one entry per token position.

        Position ``t`` maps to ``page * P + t % P``; positions in released
        pages are ``-1``.
        """
        out = []
        for p in self.block_row(rid):
            if p < 0:
                out.extend([-1] * self.page)
            else:
                out.extend(p * self.page + j for j in range(self.page))
        return out
