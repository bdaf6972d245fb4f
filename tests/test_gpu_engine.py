"""PagedKVCache.decode_step (the per-step driver) against the oracle.

Host-resident and device-resident inputs and outputs, a sliding window whose
trims release pages during the steps, and a fork whose first append copies
the shared tail page. Slots, tables and page counts bit-exact; outputs within
2e-2 (bf16)."""

import math

import numpy as np
import pytest
import torch

from gpu_harness import OracleSession, close
from libbuild import ensure_built
from paged_decode_attention_store_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def kb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_built()


@pytest.mark.parametrize("window,host_io,sinks", [(0, True, 0), (40, True, 0), (40, False, 0), (40, True, 2),
                                                  (40, False, 20)])
def test_decode_step_matches_the_oracle(kb, window, host_io, sinks):
    from paged_decode_attention_store_gb300.engine import PagedKVCache

    Hq, Hkv, D, P, seed = 32, 8, 128, 16, 71
    lengths = [300, 17, 64, 5]
    B, steps = len(lengths), 24
    num_pages = sum(-(-(L + steps) // P) for L in lengths) + 16
    order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
    w = wl.Workload("engine", "bf16", Hq, Hkv, D, P, 1, num_pages, order, lengths, window=window,
                    scale=1.0 / math.sqrt(D))
    cache = PagedKVCache(num_pages, P, Hkv, D, 1, "bf16", max_requests=B + 1, max_seq_len=512, free_stack=order,
                         device=DEV)
    orc = OracleSession(w, B + 1, seed=seed)
    # prefill requests 0..2 through the driver; request 3 is forked from 1 and then grows
    for b in range(3):
        cache.new(b)
        orc.new(b)
        slots = cache.append([b] * lengths[b])
        k, v = wl.kv_rows(seed, 0, b, list(range(lengths[b])), Hkv, D, device=DEV)
        cache.store(0, k, v, slots)
        orc.append([b] * lengths[b], list(range(lengths[b])))
        if window:
            cache.trim(b, max(0, lengths[b] + 1 - (window - sinks)), sinks=sinks)
            orc.trim(b, max(0, lengths[b] + 1 - (window - sinks)), sinks=sinks)
    cache.fork(1, 3)
    orc.fork(1, 3)
    rids = np.arange(B, dtype=np.int32)
    lens = [300, 17, 64, 17]
    for step in range(1, steps + 1):
        q = wl.q_rows(seed, step, 0, list(range(B)), Hq, D, device=DEV)
        k, v = wl.kv_rows(seed, 0, list(range(B)), lens, Hkv, D, device=DEV)
        if host_io:
            qi, ki, vi = (x.cpu().pin_memory() for x in (q, k, v))
            out = torch.empty((B, Hq, D), dtype=torch.bfloat16, pin_memory=True)
        else:
            qi, ki, vi = q, k, v
            out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
        cache.decode_step(rids, [qi], [ki], [vi], [out], window, w.scale, sinks=sinks)
        assert orc.append(list(range(B)), lens) is not None
        lens = [L + 1 for L in lens]
        got = out.float().cpu().numpy()
        for b in range(B):
            ref = orc.attend(0, b, lens[b], window, step=step, sinks=sinks)
            close(got[b], ref, "bf16", f"step {step} request {b}")
        if window:
            for b in range(B):
                orc.trim(b, max(0, lens[b] + 1 - (window - sinks)), sinks=sinks)
        assert cache.host.used() == orc.pt.used()
        assert cache.lengths[:B].tolist() == lens
    assert cache.copies == 1  # request 3's first append copied the shared tail page
    tab = cache.table.cpu().numpy()
    for b in range(B):
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    cache.check()


@pytest.mark.parametrize("window,sinks,host_io,mode", [(0, 0, True, "block"), (40, 2, True, "block"),
                                                        (0, 0, False, "raw"), (40, 0, False, "block"),
                                                        (0, 0, "reuse", "block"), (40, 2, "reuse", "raw")])
def test_device_bookkeeping_decode_step_matches_the_oracle(kb, window, sinks, host_io, mode):
    """DevicePagedKVCache: pages chosen on the device each step (one native
    call with host or device buffers); outputs, slots, tables and the device
    free list against the oracle. With ``reuse`` the steps alternate between
    two fixed sets of pinned buffers, refilled each step, as a caller reuses
    its staging buffers."""
    from paged_decode_attention_store_gb300.engine import DevicePagedKVCache

    Hq, Hkv, D, P, seed = 32, 8, 128, 16, 73
    lengths = [300, 17, 64, 5, 1000]
    B, steps = len(lengths), 20
    num_pages = sum(-(-(L + steps) // P) for L in lengths) + 8
    order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
    w = wl.Workload("devstep", "bf16", Hq, Hkv, D, P, 1, num_pages, order, lengths, window=window, sinks=sinks,
                    scale=1.0 / math.sqrt(D))
    cache = DevicePagedKVCache(num_pages, P, Hkv, D, 1, "bf16", max_requests=B, table_mode=mode,
                               max_seq_len=1100, free_stack=order, device=DEV)
    orc = OracleSession(w, B, seed=seed, mode=mode, raw_from_pages=True)
    cache.new(range(B))
    for b in range(B):
        orc.new(b)
    slots = cache.append(list(range(B)), counts=lengths)
    rr = [b for b in range(B) for _ in range(lengths[b])]
    pp = [t for L in lengths for t in range(L)]
    k, v = wl.kv_rows(seed, 0, rr, pp, Hkv, D, device=DEV)
    cache.store(0, k, v, slots)
    assert slots.cpu().tolist() == orc.append(rr, pp)
    if window:
        cache.trim(list(range(B)), window, sinks)
        for b in range(B):
            orc.trim(b, max(0, lengths[b] + 1 - (window - sinks)), sinks=sinks)
    rids = torch.arange(B, dtype=torch.int32, device=DEV)
    lens = list(lengths)
    sets = [[torch.empty(shape, dtype=torch.bfloat16, pin_memory=True) for shape in
             ((B, Hq, D), (B, Hkv, D), (B, Hkv, D), (B, Hq, D))] for _ in range(2)]
    for step in range(1, steps + 1):
        q = wl.q_rows(seed, step, 0, list(range(B)), Hq, D, device=DEV)
        k, v = wl.kv_rows(seed, 0, list(range(B)), lens, Hkv, D, device=DEV)
        if host_io == "reuse":
            qh, kh, vh, out = sets[step % 2]
            for dst, src in ((qh, q), (kh, k), (vh, v)):
                dst.copy_(src)
            cache.decode_step_host(rids, [qh], [kh], [vh], [out], window, w.scale, sinks=sinks)
        elif host_io:
            qh, kh, vh = (x.cpu().pin_memory() for x in (q, k, v))
            out = torch.empty((B, Hq, D), dtype=torch.bfloat16, pin_memory=True)
            cache.decode_step_host(rids, [qh], [kh], [vh], [out], window, w.scale, sinks=sinks)
        else:
            out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
            cache.decode_step(rids, [q], [k], [v], [out], window, w.scale, sinks=sinks)
        want_slots = orc.append(list(range(B)), lens)
        scratch = cache._staging[(B, Hq)][4] if host_io else cache._scratch[B]
        assert scratch[:B].cpu().tolist() == want_slots, f"step {step}: slots"
        lens = [L + 1 for L in lens]
        got = out.float().cpu().numpy()
        for b in range(B):
            close(got[b], orc.attend(0, b, lens[b], window, step=step, sinks=sinks), "bf16", f"step {step} request {b}")
        if window:
            for b in range(B):
                orc.trim(b, max(0, lens[b] + 1 - (window - sinks)), sinks=sinks)
    torch.cuda.synchronize()
    free, ref, lens_d, dropped, _ = cache.pages.snapshot()
    assert free == orc.pt.free and ref == orc.pt.ref
    assert lens_d[:B] == lens and dropped[:B] == [orc.pt.dropped[b] for b in range(B)]
    tab = cache.table.cpu().numpy()
    for b in range(B):
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    cache.check()


@pytest.mark.parametrize("M,mode", [(4, "block"), (3, "raw")])
def test_device_verify_step_matches_the_oracle(kb, M, mode):
    """DevicePagedKVCache.verify_step_host: the M drafts of every request
    appended, stored and verified with the page bookkeeping on the device,
    then the rejected drafts rewound, in one native call with host buffers.
    Outputs of every query against the oracle's verify positions; slots,
    tables and the device free list bit-exact after every step."""
    import random

    import oracle.attention as OA
    from paged_decode_attention_store_gb300.engine import DevicePagedKVCache

    Hq, Hkv, D, P, seed = 32, 8, 128, 16, 79
    lengths = [300, 17, 64, 5, 1000]
    B, steps = len(lengths), 8
    num_pages = sum(-(-(L + steps * M) // P) for L in lengths) + 8
    order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
    w = wl.Workload("devverify", "bf16", Hq, Hkv, D, P, 1, num_pages, order, lengths, scale=1.0 / math.sqrt(D))
    cache = DevicePagedKVCache(num_pages, P, Hkv, D, 1, "bf16", max_requests=B, table_mode=mode,
                               max_seq_len=1200, free_stack=order, device=DEV)
    orc = OracleSession(w, B, seed=seed, mode=mode, raw_from_pages=True)
    cache.new(range(B))
    for b in range(B):
        orc.new(b)
    slots = cache.append(list(range(B)), counts=lengths)
    rr = [b for b in range(B) for _ in range(lengths[b])]
    pp = [t for L in lengths for t in range(L)]
    k, v = wl.kv_rows(seed, 0, rr, pp, Hkv, D, device=DEV)
    cache.store(0, k, v, slots)
    assert slots.cpu().tolist() == orc.append(rr, pp)
    rids = torch.arange(B, dtype=torch.int32, device=DEV)
    R = random.Random(seed)
    lens = list(lengths)
    for step in range(1, steps + 1):
        rr = [b for b in range(B) for _ in range(M)]
        pos = [L + j for L in lens for j in range(M)]
        q = torch.stack([wl.q_rows(seed, step * M + j, 0, list(range(B)), Hq, D) for j in range(M)], dim=1)
        k, v = wl.kv_rows(seed, 0, rr, pos, Hkv, D)
        qh, kh, vh = (x.contiguous().pin_memory() for x in (q, k, v))
        out = torch.empty((B, M, Hq, D), dtype=torch.bfloat16, pin_memory=True)
        back = [R.randrange(0, M + 1) for _ in range(B)]
        cache.verify_step_host(rids, [qh], [kh], [vh], back, [out], 0, w.scale)
        want_slots = orc.append(rr, pos)
        scratch = cache._staging[("verify", B, M, Hq)][4]
        assert scratch[:B * M].cpu().tolist() == want_slots, f"step {step}: slots"
        ctx = [L + M for L in lens]
        got = out.float().numpy()
        for b in range(B):
            for j, ps in enumerate(OA.verify_positions(ctx[b], M, None)):
                ref = OA.attend_request(orc.stores[0], q[b, j].float().numpy(),
                                        [s for p in ps for s in orc.slots(b, p, p + 1)], w.scale)
                close(got[b, j], ref, "bf16", f"step {step} request {b} query {j}")
        for b in range(B):
            orc.pt.rewind(b, back[b])
        lens = [c - nb for c, nb in zip(ctx, back)]
    torch.cuda.synchronize()
    free, ref, lens_d, _, _ = cache.pages.snapshot()
    assert free == orc.pt.free and ref == orc.pt.ref
    assert lens_d[:B] == lens
    tab = cache.table.cpu().numpy()
    for b in range(B):
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    cache.check()


@pytest.mark.parametrize("window,sinks", [(0, 0), (100, 4)])
def test_prefill_step_matches_the_oracle(kb, window, sinks):
    """PagedKVCache.prefill_step (the per-step driver of chunked prefill, host
    bookkeeping) with pinned host buffers: each request's chunk is appended,
    stored and attended at once; every query's output against the oracle
    (query j of a chunk attends what a one-token step with context
    prefix + j + 1 attends), slots and table rows bit-exact. Two chunks, so
    the second attends the first."""
    import oracle.attention as OA
    from paged_decode_attention_store_gb300.engine import PagedKVCache

    Hq, Hkv, D, P, seed, C = 32, 8, 128, 16, 83, 48
    prefixes = [100, 0, 37]
    B, chunks = len(prefixes), 2
    num_pages = sum(-(-(L + chunks * C) // P) for L in prefixes) + 8
    order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
    w = wl.Workload("prefillstep", "bf16", Hq, Hkv, D, P, 1, num_pages, order, prefixes, window=window, sinks=sinks,
                    scale=1.0 / math.sqrt(D))
    cache = PagedKVCache(num_pages, P, Hkv, D, 1, "bf16", max_requests=B, max_seq_len=512, free_stack=order,
                         device=DEV)
    orc = OracleSession(w, B, seed=seed)
    for b in range(B):
        cache.new(b)
        orc.new(b)
        if prefixes[b]:
            slots = cache.append([b] * prefixes[b])
            k, v = wl.kv_rows(seed, 0, b, list(range(prefixes[b])), Hkv, D, device=DEV)
            cache.store(0, k, v, slots)
            assert slots.cpu().tolist() == orc.append([b] * prefixes[b], list(range(prefixes[b])))
    lens = list(prefixes)
    rids = np.arange(B, dtype=np.int32)
    for step in range(1, chunks + 1):
        rr = [b for b in range(B) for _ in range(C)]
        pos = [L + j for L in lens for j in range(C)]
        q = torch.stack([wl.q_rows(seed, step * C + j, 0, list(range(B)), Hq, D) for j in range(C)], dim=1)
        k, v = wl.kv_rows(seed, 0, rr, pos, Hkv, D)
        qh, kh, vh = (x.contiguous().pin_memory() for x in (q, k, v))
        out = torch.empty((B, C, Hq, D), dtype=torch.bfloat16, pin_memory=True)
        cache.prefill_step(rids, [qh], [kh], [vh], [out], window, w.scale, sinks=sinks)
        assert orc.append(rr, pos) is not None
        lens = [L + C for L in lens]
        assert cache.lengths[:B].tolist() == lens
        got = out.float().numpy()
        for b in range(B):
            for j, ps in enumerate(OA.verify_positions(lens[b], C, window if window > 0 else None, sinks)):
                ref = OA.attend_request(orc.stores[0], q[b, j].float().numpy(),
                                        [s for p in ps for s in orc.slots(b, p, p + 1)], w.scale)
                close(got[b, j], ref, "bf16", f"chunk {step} request {b} query {j}")
    tab = cache.table.cpu().numpy()
    for b in range(B):
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    cache.check()
