"""Device-side page allocation (kvp_dev_*) against the oracle's page table.

Random batches of new / append (several rows per request) / fork / trim
(with sink pages) / rewind / release run on the device and on the oracle
(chapter 15's page table, restated in oracle/pagetable.py) from the same
free-list order. After every batch the device state read back must equal
the oracle's bit for bit: the free list, every reference count, lengths,
released-page counts and the table rows (block ids, or token slots for a
raw-location table); the slots of the appended rows and the copy-on-write
pairs must equal the oracle's in call order. A batch the pool cannot serve
must fail whole (KVP_ERR_OUT_OF_PAGES) and change nothing.
"""

import copy
import random

import pytest
import torch

from libbuild import ensure_built
from oracle.pagetable import OutOfPages, PageTable

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def kb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_built()


def _i32(xs):
    return torch.tensor(list(xs), dtype=torch.int32, device=DEV)


def _compare(dev, opt, live, mode, P):
    stack, ref, lens, dropped, _ = dev.snapshot()
    assert stack == opt.free, "free list"
    assert ref == opt.ref, "reference counts"
    tab = dev.table.cpu()
    for r in live:
        assert lens[r] == opt.length[r] and dropped[r] == opt.dropped[r], f"request {r} length / released pages"
        row = opt.block_row(r) if mode == "block" else opt.raw_row(r)
        assert tab[r, :len(row)].tolist() == row, f"table row {r}"


@pytest.mark.parametrize("seed", range(8))
def test_device_pages_match_the_oracle(kb, seed):
    R = random.Random(seed)
    P = [1, 4, 16, 3][seed % 4]
    mode = "block" if seed < 4 else "raw"
    n_pages, max_req = (48 if P >= 4 else 160), 12
    cap = 600  # positions a request may reach
    cols = -(-cap // P) if mode == "block" else -(-cap // P) * P
    table = torch.full((max_req, cols), -1, dtype=torch.int32, device=DEV)
    order = list(range(n_pages))
    R.shuffle(order)
    dev = kb.DevicePages(n_pages, P, max_req, table, kb.KVP_RAW_LOCATIONS if mode == "raw" else kb.KVP_BLOCK_TABLE,
                         free_stack=order, device=DEV)
    opt = PageTable(n_pages, P, free_order=order)
    live, sinks = [], {}
    out_loc = torch.empty(4 * max_req * 6, dtype=torch.int32, device=DEV)
    cs = torch.empty(max_req, dtype=torch.int32, device=DEV)
    cd = torch.empty(max_req, dtype=torch.int32, device=DEV)
    nc = torch.zeros(1, dtype=torch.int32, device=DEV)
    for step in range(160):
        op = R.choice(["append"] * 5 + ["new", "fork", "trim", "trim", "rewind", "rewind", "release"])
        free = [r for r in range(max_req) if r not in live]
        if op == "new" and free:
            rids = free[:R.randrange(1, min(3, len(free)) + 1)]
            dev.new(_i32(rids))
            for r in rids:
                opt.new(r)
                sinks[r] = R.choice([0, 0, 1, 5])
            live += rids
        elif op == "append" and live:
            rids = R.sample(live, R.randrange(1, len(live) + 1))
            counts = [R.randrange(0, 6) for _ in rids]
            if any(opt.length[r] + c > cap for r, c in zip(rids, counts)):
                continue
            snap = copy.deepcopy(opt)
            try:
                want = [opt.append(r) for r, c in zip(rids, counts) for _ in range(c)]
            except OutOfPages:
                opt = snap
                dev.append(_i32(rids), out_loc, cs, cd, nc, counts=_i32(counts))
                assert dev.sync_error() == kb.KVP_ERR_OUT_OF_PAGES
            else:
                dev.append(_i32(rids), out_loc, cs, cd, nc, counts=_i32(counts))
                assert dev.sync_error() == 0
                assert out_loc[:len(want)].tolist() == [w["slot"] for w in want]
                cows = [w["cow"] for w in want if w["cow"] is not None]
                n = int(nc.item())
                assert list(zip(cs[:n].tolist(), cd[:n].tolist())) == cows
        elif op == "fork" and live and free:
            k = min(len(free), R.randrange(1, 3))
            src = [R.choice(live) for _ in range(k)]
            dst = free[:k]
            dev.fork(_i32(src), _i32(dst))
            for a, b in zip(src, dst):
                opt.fork(a, b)
                sinks[b] = sinks[a]
            live += dst
        elif op == "trim" and live:
            rids = R.sample(live, R.randrange(1, len(live) + 1))
            S = R.choice([0, 1, 5])
            rids = [r for r in rids if opt.dropped[r] == 0 or opt.sinks[r] == -(-S // P)]
            if not rids:
                continue
            keep = [R.randrange(0, opt.length[r] + 1) for r in rids]
            dev.trim(_i32(rids), _i32(keep), sinks=S)
            for r, k in zip(rids, keep):
                if S:
                    opt.trim(r, k, sink_rows=S)
                else:
                    opt.trim(r, k)
        elif op == "rewind" and live:
            rids = R.sample(live, R.randrange(1, len(live) + 1))
            back = []
            for r in rids:  # no rewind into released rows (the oracle refuses it)
                floor = (opt.sinks[r] + opt.dropped[r]) * P if opt.dropped[r] else 0
                back.append(R.randrange(0, min(opt.length[r] - floor, 2 * P + 3) + 1))
            dev.rewind(_i32(rids), _i32(back))
            for r, nb in zip(rids, back):
                opt.rewind(r, nb)
        elif op == "release" and live:
            rids = R.sample(live, R.randrange(1, min(3, len(live)) + 1))
            dev.release(_i32(rids))
            for r in rids:
                opt.release(r)
                live.remove(r)
        assert dev.sync_error() == 0, f"step {step} ({op})"
        _compare(dev, opt, live, mode, P)


def test_device_append_refuses_bad_calls(kb):
    P, n_pages = 4, 8
    table = torch.full((4, 8), -1, dtype=torch.int32, device=DEV)
    dev = kb.DevicePages(n_pages, P, 4, table, kb.KVP_BLOCK_TABLE, device=DEV)
    dev.new(_i32([0, 1]))
    out = torch.empty(64, dtype=torch.int32, device=DEV)
    cs, cd, nc = (torch.zeros(4, dtype=torch.int32, device=DEV) for _ in range(3))
    before = dev.snapshot()
    dev.append(_i32([0, 0]), out, cs, cd, nc)  # the same request twice in one call
    assert dev.sync_error() == kb.KVP_ERR_INVALID_ARG and dev.snapshot() == before
    dev.append(_i32([0, 7]), out, cs, cd, nc)  # no such request
    assert dev.sync_error() == kb.KVP_ERR_INVALID_ARG and dev.snapshot() == before
    dev.append(_i32([0, 1]), out[:3], cs, cd, nc, counts=_i32([2, 2]))  # four slots, room for three
    assert dev.sync_error() == kb.KVP_ERR_INVALID_ARG and dev.snapshot() == before
    dev.append(_i32([0, 1]), out, cs, cd, nc, counts=_i32([33, 1]))  # a row holds 8 pages of 4: 32 positions
    assert dev.sync_error() == kb.KVP_ERR_INVALID_ARG and dev.snapshot() == before
    dev.append(_i32([0, 1]), out, cs, cd, nc, counts=_i32([20, 16]))  # 9 pages wanted, 8 in the pool
    assert dev.sync_error() == kb.KVP_ERR_OUT_OF_PAGES and dev.snapshot() == before
    dev.append(_i32([0, 1]), out, cs, cd, nc, counts=_i32([16, 16]))  # exactly the pool
    assert dev.sync_error() == 0 and dev.snapshot()[0] == []


def test_device_rewind_refuses_released_rows(kb):
    """A rewind below the rows a window released, or of more rows than a
    request holds, fails whole and changes nothing."""
    P, n_pages = 4, 16
    table = torch.full((2, 16), -1, dtype=torch.int32, device=DEV)
    dev = kb.DevicePages(n_pages, P, 2, table, kb.KVP_BLOCK_TABLE, device=DEV)
    dev.new(_i32([0, 1]))
    out = torch.empty(64, dtype=torch.int32, device=DEV)
    cs, cd, nc = (torch.zeros(2, dtype=torch.int32, device=DEV) for _ in range(3))
    dev.append(_i32([0, 1]), out, cs, cd, nc, counts=_i32([14, 6]))
    dev.trim(_i32([0]), _i32([9]))  # request 0 lets go of pages 0 and 1 (rows 0..7)
    assert dev.sync_error() == 0
    before = dev.snapshot()
    dev.rewind(_i32([1, 0]), _i32([1, 7]))  # request 0 would keep 7 rows, inside its released pages
    assert dev.sync_error() == kb.KVP_ERR_INVALID_ARG and dev.snapshot() == before
    dev.rewind(_i32([1]), _i32([7]))  # request 1 holds 6 rows
    assert dev.sync_error() == kb.KVP_ERR_INVALID_ARG and dev.snapshot() == before
    dev.rewind(_i32([0, 1]), _i32([6, 6]))  # down to row 8 and to nothing: allowed
    assert dev.sync_error() == 0
    _, _, lens, _, _ = dev.snapshot()
    assert lens[:2] == [8, 0]
