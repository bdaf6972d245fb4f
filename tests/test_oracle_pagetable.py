"""Pins of the oracle's block-table bookkeeping (CPU only).

Expected values come from the pages (golden files) or from closed forms the
pages state; the mutation tests plant the chapter's one-line mistakes in
copies of the oracle and require the pins to notice each one.
"""

import random

import pytest

import oracle_pins as op
from oracle.pagetable import OutOfPages, PageTable


def test_example_a_trace():
    assert op.check_example_a(PageTable, OutOfPages) == []


def test_pages_in_use_of_the_32_step_run():
    assert op.check_pages_in_use(PageTable) == []


def test_exact_page_count_every_step():
    assert op.check_exact_counts(PageTable) == []


@pytest.mark.parametrize("seed", range(6))
def test_shadow_model_chapter_seeds(seed):
    assert op.check_shadow(PageTable, OutOfPages, seed) == []


def test_shadow_model_thousands_of_operations():
    # 40 more sequences of 400 operations (16,000 operations), larger pools too.
    problems = []
    for seed in range(100, 120):
        problems += op.check_shadow(PageTable, OutOfPages, seed)
    for seed in range(200, 220):
        problems += op.check_shadow(PageTable, OutOfPages, seed, n_pages=64, page=3, max_live=8)
    assert problems == []


def test_exhaustion_leaves_state_unchanged():
    assert op.check_exhaustion(PageTable, OutOfPages) == []


def test_paged_gather_equals_plain_list():
    assert op.check_paged_equals_plain(PageTable) == []


def test_prefix_sharing_table():
    assert op.check_prefix_sharing(PageTable) == []


def test_admission_table():
    assert op.check_admission(PageTable, OutOfPages) == []


def test_translate_closed_form():
    """Position t lives in logical page t // P at offset t % P; outside
    [0, length) is an error ("PagedAttention block allocator", section
    "Sequence block table")."""
    R = random.Random(5)
    for P in (1, 3, 4, 16):
        order = list(range(50))
        R.shuffle(order)
        pt = PageTable(50, P, free_order=order)
        pt.new(0)
        n = R.randrange(1, 50 * P // 2)
        for i in range(n):
            pt.append(0, i)
        popped = list(reversed(order))[: -(-n // P)]  # pages in hand-out order
        for t in range(n):
            assert pt.translate(0, t) == (popped[t // P], t % P)
            assert pt.slot(0, t) == popped[t // P] * P + t % P
        for bad in (-1, n, n + P):
            with pytest.raises(IndexError):
                pt.translate(0, bad)


def test_block_row_holes_and_raw_expansion():
    pt = PageTable(16, 4)
    pt.new(0)
    for i in range(14):
        pt.append(0, i)
    released = pt.trim(0, 9)  # pages 0 and 1 hold only rows < 9? page 1 holds 4..7 -> released
    assert released == [0, 1]
    row = pt.block_row(0)
    assert row[:2] == [-1, -1] and len(row) == 4
    raw = pt.raw_row(0)
    assert raw[:8] == [-1] * 8
    for t in range(8, 14):
        assert raw[t] == row[t // 4] * 4 + t % 4 == pt.slot(0, t)


@pytest.mark.parametrize("W,P", [(4096, 16), (100, 16), (7, 1), (33, 8), (16, 16)])
def test_window_footprint_bound_long_run(W, P):
    """Footprint after each trimmed step never exceeds ceil((W-1)/P)+1 pages,
    and one more transiently (chapter 15, section "The problem" and "Tests")."""
    bound = -(-(W - 1) // P) + 1
    pt = PageTable(bound + 8, P)
    pt.new(0)
    for L in range(1, 3 * W + 5 * P):
        pt.append(0, None)
        assert pt.used() <= bound + 1
        pt.trim(0, max(0, L + 1 - W))
        assert pt.used() <= bound


# ---------------------------------------------------------------------------
# Mutation tests: the chapter's one-line mistakes, planted in oracle copies.
# ---------------------------------------------------------------------------
class FreedNotReturned(PageTable):
    def _unref(self, p):
        self.ref[p] -= 1


class FreedWhileShared(PageTable):
    def _unref(self, p):
        self.ref[p] -= 1
        if self.ref[p] <= 1 and p not in self.free:
            self.free.append(p)


class ForkNotCounting(PageTable):
    def fork(self, src, dst):
        self.table[dst] = list(self.table[src])
        self.length[dst] = self.length[src]
        self.dropped[dst] = self.dropped[src]


class NoCopyOnWrite(PageTable):
    def append(self, rid, row=None):
        i = self.length[rid]
        off = i % self.page
        t = self.table[rid]
        if off == 0:
            t.append(self._alloc())
        self.pool[t[-1]][off] = row
        self.length[rid] = i + 1
        return {"slot": t[-1] * self.page + off, "cow": None}


class _CowVariant(PageTable):
    empty_copy = False
    keep_ref = False

    def append(self, rid, row=None):
        i = self.length[rid]
        off = i % self.page
        t = self.table[rid]
        if off == 0:
            t.append(self._alloc())
        elif self.ref[t[-1]] > 1:
            q = self._alloc()
            self.pool[q] = [None] * self.page if self.empty_copy else list(self.pool[t[-1]])
            if not self.keep_ref:
                self._unref(t[-1])
            t[-1] = q
        self.pool[t[-1]][off] = row
        self.length[rid] = i + 1
        return {"slot": t[-1] * self.page + off, "cow": None}


class EmptyCopy(_CowVariant):
    empty_copy = True


class CopyKeepsReference(_CowVariant):
    keep_ref = True


class OffsetPagePlusOne(PageTable):
    def append(self, rid, row=None):
        i = self.length[rid]
        off = i % (self.page + 1)
        t = self.table[rid]
        if off == 0:
            t.append(self._alloc())
        elif self.ref[t[-1]] > 1:
            q = self._alloc()
            self.pool[q] = list(self.pool[t[-1]])
            self._unref(t[-1])
            t[-1] = q
        self.pool[t[-1]][off % self.page] = row
        self.length[rid] = i + 1
        return {"slot": t[-1] * self.page + off, "cow": None}


class LookupIgnoresDropped(PageTable):
    def rows(self, rid, lo, hi):
        t = self.table[rid]
        return [self.pool[t[min(i // self.page, len(t) - 1)]][i % self.page] for i in range(lo, hi)]


class TrimTooMuch(PageTable):
    def trim(self, rid, keep_from):
        t = self.table[rid]
        while t and self.dropped[rid] * self.page < keep_from:
            self._unref(t.pop(0))
            self.dropped[rid] += 1
        return []

    def rows(self, rid, lo, hi):
        lo = max(lo, self.dropped[rid] * self.page)
        return super().rows(rid, lo, hi)


class TrimTooLittle(PageTable):
    def trim(self, rid, keep_from):
        t = self.table[rid]
        while t and (self.dropped[rid] + 1) * self.page < keep_from:
            self._unref(t.pop(0))
            self.dropped[rid] += 1
        return []


class ReleaseForgets(PageTable):
    def release(self, rid):
        self.table.pop(rid)
        del self.length[rid]
        del self.dropped[rid]


class ExhaustionUnreported(PageTable):
    def _alloc(self):
        if not self.free:
            return 0
        return super()._alloc()


MUTANTS = [FreedNotReturned, FreedWhileShared, ForkNotCounting, NoCopyOnWrite, EmptyCopy,
           CopyKeepsReference, OffsetPagePlusOne, LookupIgnoresDropped, TrimTooMuch,
           TrimTooLittle, ReleaseForgets, ExhaustionUnreported]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_bookkeeping_mutant_is_caught(mutant):
    try:
        problems = op.all_bookkeeping_problems(mutant, OutOfPages)
    except Exception as e:  # a crash is a catch too
        problems = [repr(e)]
    assert problems, f"{mutant.__name__} survived every pin"
