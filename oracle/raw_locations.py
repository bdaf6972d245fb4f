"""Raw token-location page table oracle (test infrastructure only; see ``oracle``).

Restates the layout and allocation steps of the mini-sglang code series,
part 4 (jaehun.me), sections "표에는 raw location이 들어간다" (the table holds
raw locations), "할당은 페이지로, 기록은 토큰으로" (allocate in pages, record
in tokens), "더미 요청이 가리키는 곳" (where the dummy request points) and
"페이지 정렬은 테스트가 지킨다" (page alignment is guarded by tests):

* the table has ``max_running_req + 1`` rows (the extra one belongs to a
  dummy request) and ``align32(min(max_seq_len, num_tokens))`` int32
  columns, zero-initialised; ``table[row][pos]`` is the flat token location
  of position ``pos`` of the request in that row, so a reader needs no
  ``page * P + offset`` arithmetic;
* the free list holds the FIRST token location of each free page
  (``page * P``);
* a request growing from ``cached_len`` to ``device_len`` needs
  ``ceil(device_len / P) - ceil(cached_len / P)`` new pages; all requests of
  one call are counted, the pages are taken in one allocation, expanded to
  token locations (``s, s+1, …, s+P-1`` per page start ``s``; identity for
  ``P = 1``) and written by ONE scatter over host-built (row, position)
  lists;
* ``num_tokens = num_pages * P`` is where the managed pages end; the pool
  holds one more page that is never handed out, and the dummy row is filled
  with ``num_tokens`` so that it points into that page.

Readings where the page is silent: the allocator body is not shown, so the
free list is read as the same stack as chapter 15's page table (the end of
the list goes out first, freed pages are pushed back on the end, in table
order); the initial order may be a seeded shuffle.
"""

from __future__ import annotations

import numpy as np

from .pagetable import OutOfPages


def align32(n: int) -> int:
    return (n + 31) // 32 * 32


def div_ceil(a: int, b: int) -> int:
    return -(-a // b)


class RawLocationTable:
    def __init__(self, num_pages: int, page_size: int, max_running_req: int,
                 max_seq_len: int, free_page_order=None):
        self.P = page_size
        self.num_pages = num_pages
        self.num_tokens = num_pages * page_size
        self.max_seq_len = min(max_seq_len, self.num_tokens)
        cols = align32(self.max_seq_len)
        self.page_table = np.zeros((max_running_req + 1, cols), dtype=np.int32)
        self.dummy_row = max_running_req
        self.page_table[self.dummy_row, :] = self.num_tokens
        order = range(num_pages - 1, -1, -1) if free_page_order is None else free_page_order
        order = [int(p) for p in order]
        if sorted(order) != list(range(num_pages)):
            raise ValueError("free_page_order must be a permutation of 0..num_pages-1")
        self.free_slots = [p * page_size for p in order]
        self.held = {}  # table row -> list of page-start locations, logical order

    def _allocate(self, n_pages: int) -> list:
        if n_pages > len(self.free_slots):
            raise OutOfPages(f"{n_pages} pages wanted, {len(self.free_slots)} free")
        return [self.free_slots.pop() for _ in range(n_pages)]

    def _page_to_token(self, page_starts: list) -> list:
        if self.P == 1:
            return list(page_starts)
        return [s + j for s in page_starts for j in range(self.P)]

    def allocate_paged(self, reqs) -> list:
        """``reqs``: iterable of ``(table_idx, cached_len, device_len)``.

        Returns the allocation info ``(table_idx, first_page, last_page)`` of
        the requests that needed pages.
        """
        needed = 0
        info = []
        for table_idx, cached_len, device_len in reqs:
            first_page = div_ceil(cached_len, self.P)
            last_page = div_ceil(device_len, self.P)
            if last_page > first_page:
                needed += last_page - first_page
                info.append((table_idx, first_page, last_page))
        if needed > 0:
            starts = self._allocate(needed)
            k = 0
            for table_idx, first_page, last_page in info:
                n = last_page - first_page
                self.held.setdefault(table_idx, []).extend(starts[k:k + n])
                k += n
            self._write_page_table(self._page_to_token(starts), info)
        return info

    def _write_page_table(self, allocated: list, info: list) -> None:
        rows, positions = [], []
        for table_idx, first_page, last_page in info:
            first_pos, last_pos = first_page * self.P, last_page * self.P
            rows.extend([table_idx] * (last_pos - first_pos))
            positions.extend(range(first_pos, last_pos))
        if len(rows) != len(allocated):
            raise AssertionError("allocated tokens and table positions differ in number")
        self.page_table[np.asarray(rows), np.asarray(positions)] = np.asarray(allocated, dtype=np.int32)

    def free_request(self, table_idx: int) -> None:
        """Return every page of a finished request to the free list."""
        for s in self.held.pop(table_idx, []):
            self.free_slots.append(s)

    def check_no_leak(self) -> None:
        """Free pages plus held pages must account for every managed page."""
        held = sum(len(v) for v in self.held.values())
        if len(self.free_slots) + held != self.num_pages:
            raise RuntimeError("a page is neither free nor held")
