"""The GPU path's host bookkeeping (C++, kvp_host_*) against the oracle (CPU).

Both start from the same free-list order and receive the same operations;
slots, block-table rows (with -1 holes), reference counts, free lists and
copy-on-write pairs must agree bit for bit after every operation. The two
share no code: the C++ side is the product, the oracle is the Python
restatement of chapter 15's page table.
"""

import random

import pytest

from libbuild import ensure_built
from oracle.pagetable import OutOfPages, PageTable


def _state_equal(host, opt, live):
    assert host.refcounts() == opt.ref
    assert host.free_list() == opt.free
    assert host.used() == opt.used()
    for rid in live:
        assert host.block_row(rid) == opt.block_row(rid)
        assert host.length(rid) == (opt.length[rid], opt.dropped[rid])


@pytest.mark.parametrize("seed", range(18))
def test_shadow_ops_match_the_oracle(seed):
    """Seeds 12-17 give each request a fixed number of attention-sink rows
    that its trims keep (chapter 15, exercise "Attention sinks")."""
    kb = ensure_built()
    R = random.Random(seed)
    n_pages, P = (24, 4) if seed < 6 or seed >= 12 else (64, R.choice([1, 3, 16]))
    sinks = {}
    order = list(range(n_pages))
    R.shuffle(order)
    host = kb.HostPageTable(n_pages, P, 16, order)
    opt = PageTable(n_pages, P, free_order=order)
    live = []
    for step in range(400):
        op = R.choice(["append"] * 6 + ["new", "fork", "trim", "release", "batch", "rewind"])
        free_rids = [r for r in range(16) if r not in live]
        if op == "new" and len(live) < 6:
            rid = free_rids[0]
            host.new(rid)
            opt.new(rid)
            live.append(rid)
            sinks[rid] = R.choice([0, 1, 2, 4, 5, 9]) if seed >= 12 else 0
        elif op in ("append", "batch") and live:
            rids = [R.choice(live) for _ in range(1 if op == "append" else R.randrange(1, 6))]
            snapshot = (opt.free[:], opt.ref[:], {r: (opt.table[r][:], opt.length[r]) for r in live})
            try:
                want = [opt.append(r) for r in rids]
            except OutOfPages:
                # the oracle ran out part way; the batch must fail whole on the host
                opt.free, opt.ref = snapshot[0], snapshot[1]
                for r, (t, L) in snapshot[2].items():
                    opt.table[r], opt.length[r] = t, L
                with pytest.raises(kb.OutOfPages):
                    host.append(rids)
            else:
                slots, writes, cows = host.append(rids)
                assert slots == [w["slot"] for w in want]
                assert cows == [w["cow"] for w in want if w["cow"] is not None]
                exp_writes = [(r, w["logical_page"], w["page"]) for r, w in zip(rids, want)
                              if w["new_page"] is not None or w["cow"] is not None]
                assert writes == exp_writes
        elif op == "fork" and live and len(live) < 6:
            src, dst = R.choice(live), free_rids[0]
            writes = host.fork(src, dst)
            opt.fork(src, dst)
            sinks[dst] = sinks[src]
            assert writes == [(dst, i, p) for i, p in enumerate(opt.block_row(dst))]
            live.append(dst)
        elif op == "trim" and live:
            rid = R.choice(live)
            k = R.randrange(0, opt.length[rid] + 1)
            writes = host.trim(rid, k, sinks=sinks[rid])
            released = opt.trim(rid, k, sink_rows=sinks[rid]) if sinks[rid] else opt.trim(rid, k)
            assert writes == [(rid, d, -1) for d in released]
        elif op == "rewind" and live:
            rid = R.choice(live)
            L, d = opt.length[rid], opt.dropped[rid]
            floor = (opt.sinks[rid] + d) * P if d else 0
            n = R.randrange(0, L - floor + 1)
            writes = host.rewind(rid, n)
            gone = opt.rewind(rid, n)
            assert writes == [(rid, g, -1) for g in gone]
            if d:  # one row past the released front is refused and changes nothing
                with pytest.raises(kb.KvpError):
                    host.rewind(rid, opt.length[rid] - floor + 1)
        elif op == "release" and live:
            rid = R.choice(live)
            host.release(rid)
            opt.release(rid)
            live.remove(rid)
        _state_equal(host, opt, live)


def test_example_a_on_the_host_bookkeeping():
    """Chapter 15, worked example A: tables and free list at every step."""
    kb = ensure_built()
    host = kb.HostPageTable(8, 4, 2)
    opt = PageTable(8, 4)
    host.new(0)
    opt.new(0)
    for L in range(1, 15):
        host.append([0])
        opt.append(0, L - 1)
        host.trim(0, max(0, L + 1 - 6))
        opt.trim(0, max(0, L + 1 - 6))
        _state_equal(host, opt, [0])
    assert [p for p in host.block_row(0) if p >= 0] == [2, 0]


def test_exhaustion_fails_whole_batch_and_changes_nothing():
    kb = ensure_built()
    host = kb.HostPageTable(3, 2, 2)
    host.new(0)
    host.append([0] * 6)
    before = (host.free_list(), host.refcounts(), host.block_row(0), host.length(0))
    with pytest.raises(kb.OutOfPages):
        host.append([0])
    assert (host.free_list(), host.refcounts(), host.block_row(0), host.length(0)) == before
    # a batch that would need two pages when one is free fails as a whole
    host2 = kb.HostPageTable(3, 2, 2)
    host2.new(0)
    host2.new(1)
    host2.append([0, 0, 0, 0])  # two pages
    snap = (host2.free_list(), host2.refcounts())
    with pytest.raises(kb.OutOfPages):
        host2.append([1, 1, 1])  # needs two pages, one free
    assert (host2.free_list(), host2.refcounts()) == snap and host2.length(1) == (0, 0)


def test_prefix_sharing_copy_on_write_counts():
    """8 prompts of 2050 tokens, 16 forks each, page 16: every fork's first
    append copies the shared tail page once (128 copies) while the prompt
    request still holds it."""
    kb = ensure_built()
    P = 16
    host = kb.HostPageTable(2000, P, 8 + 128)
    for i in range(8):
        host.new(128 + i)
        host.append([128 + i] * 2050)
    for f in range(128):
        host.fork(128 + f // 16, f)
    _, writes, cows = host.append(list(range(128)))
    assert len(cows) == 128 and len(writes) == 128
    # each copy's destination is the page its table write installs
    assert [c[1] for c in cows] == [w[2] for w in writes]
    for i in range(8):
        host.release(128 + i)
    ref = host.refcounts()
    # 128 full prompt pages per prompt stay shared by 16 forks; tails are private
    shared = [p for p in range(2000) if ref[p] == 16]
    assert len(shared) == 8 * 128
    assert host.used() == 8 * 128 + 128
