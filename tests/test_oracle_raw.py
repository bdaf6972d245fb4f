"""Pins of the oracle's raw token-location page table (CPU only).

Anchors: the layout and the dummy row the mini-sglang code series (part 4)
states, brute-force page counting on tiny inputs, the page-alignment and
no-leak invariants its tests guard, the identity expansion at page size 1,
and agreement with an independent procedure (chapter 15's page table driven
token by token, then expanded) under the same free-list order.
"""

import random

import numpy as np
import pytest

from oracle.pagetable import OutOfPages, PageTable
from oracle.raw_locations import RawLocationTable, align32, div_ceil


def test_layout_and_dummy_row():
    # The large-batch layout: 256 running requests + 1 dummy row, 16384 columns.
    t = RawLocationTable(num_pages=2000, page_size=16, max_running_req=256, max_seq_len=16384)
    assert t.page_table.shape == (257, 16384) and t.page_table.dtype == np.int32
    assert np.all(t.page_table[256] == 2000 * 16)  # the first slot of the extra page
    assert np.all(t.page_table[:256] == 0)
    # max_seq_len is clipped by the managed tokens, then aligned to 32.
    t2 = RawLocationTable(num_pages=10, page_size=3, max_running_req=2, max_seq_len=999)
    assert t2.page_table.shape == (3, align32(30)) == (3, 32)


def test_page_count_matches_brute_force():
    R = random.Random(1)
    for _ in range(300):
        P = R.choice([1, 2, 4, 16])
        cached = R.randrange(0, 40)
        device = cached + R.randrange(0, 40)
        brute = len({t // P for t in range(device)}) - len({t // P for t in range(cached)})
        t = RawLocationTable(128, P, 1, 128 * P)
        # Bring the request to `cached` first, then grow it.
        t.allocate_paged([(0, 0, cached)])
        free_before = len(t.free_slots)
        t.allocate_paged([(0, cached, device)])
        assert free_before - len(t.free_slots) == brute == div_ceil(device, P) - div_ceil(cached, P)


def test_page_size_one_is_identity_and_alignment_holds():
    R = random.Random(2)
    for P in (1, 4, 16):
        order = list(range(40))
        R.shuffle(order)
        t = RawLocationTable(40, P, 4, 40 * P, free_page_order=order)
        lens = [0, 0, 0, 0]
        for _ in range(30):
            reqs = []
            for r in range(4):
                grow = R.randrange(0, 2 * P + 1)
                if sum(div_ceil(x, P) for x in lens) + 4 * 3 > 40:
                    grow = 0
                reqs.append((r, lens[r], lens[r] + grow))
                lens[r] += grow
            t.allocate_paged(reqs)
        for r in range(4):
            row = t.page_table[r, : div_ceil(lens[r], P) * P]
            starts = row[::P]
            assert np.all(starts % P == 0), "a page does not start on a page boundary"
            for j in range(P):
                assert np.array_equal(row[j::P], starts + j)
            if P == 1:
                assert list(row) == t.held[r]
        t.check_no_leak()
        for r in range(4):
            t.free_request(r)
        t.check_no_leak()
        assert sorted(t.free_slots) == [p * P for p in range(40)]


def test_matches_block_table_expansion():
    """P3's procedure (count pages per call, one allocation, one scatter)
    gives the same table as chapter 15's page table appending token by token
    and expanding each page to its token locations, when both start from the
    same free list and serve requests in the same order."""
    R = random.Random(3)
    for P in (1, 4, 16):
        order = list(range(1200))
        R.shuffle(order)
        raw = RawLocationTable(1200, P, 6, 1200 * P, free_page_order=order)
        pt = PageTable(1200, P, free_order=order)
        lens = [0] * 6
        for r in range(6):
            pt.new(r)
        for _ in range(40):
            reqs = []
            for r in range(6):
                grow = R.randrange(0, 9)
                for _ in range(grow):
                    pt.append(r)
                reqs.append((r, lens[r], lens[r] + grow))
                lens[r] += grow
            raw.allocate_paged(reqs)
        for r in range(6):
            n = len(pt.block_row(r)) * P
            assert list(raw.page_table[r, :n]) == pt.raw_row(r)


def test_exhaustion_changes_nothing():
    t = RawLocationTable(4, 2, 2, 8)
    t.allocate_paged([(0, 0, 5)])  # 3 pages
    snap = (t.page_table.copy(), list(t.free_slots))
    with pytest.raises(OutOfPages):
        t.allocate_paged([(1, 0, 4)])  # 2 pages wanted, 1 free
    assert np.array_equal(t.page_table, snap[0]) and t.free_slots == snap[1]


# Planted mistakes: each must fail one of the checks above.
class NoOffsets(RawLocationTable):
    def _page_to_token(self, page_starts):
        return [s for s in page_starts for _ in range(self.P)]


class FloorCount(RawLocationTable):
    def allocate_paged(self, reqs):
        return super().allocate_paged([(i, c - (c % self.P if c % self.P else 0), d) for i, c, d in reqs])


class DummyOutside(RawLocationTable):
    def __init__(self, *a, **k):
        super().__init__(*a, **k)
        self.page_table[self.dummy_row, :] = self.num_tokens + self.P


@pytest.mark.parametrize("mutant", [NoOffsets, FloorCount, DummyOutside], ids=lambda m: m.__name__)
def test_raw_mutant_is_caught(mutant, monkeypatch):
    import test_oracle_raw as me
    monkeypatch.setattr(me, "RawLocationTable", mutant)
    caught = False
    for check in (test_layout_and_dummy_row, test_page_count_matches_brute_force,
                  test_page_size_one_is_identity_and_alignment_holds, test_matches_block_table_expansion):
        try:
            check()
        except (AssertionError, OutOfPages, RuntimeError, ValueError):
            caught = True
    assert caught, f"{mutant.__name__} survived"
