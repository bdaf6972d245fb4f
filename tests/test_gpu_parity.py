"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: store_cache writes, slots, page-table contents, copied pages and
gathered indices. Attention outputs: max |gpu - oracle| <= 1e-5 for fp32
caches and <= 2e-2 for bf16 caches (oracle in float64 over the same
bf16-rounded inputs). Sizes are small enough for the oracle to finish in
seconds yet span many 16-token stages, split requests and ragged tails.
"""

import math
import random

import numpy as np
import pytest
import torch

from gpu_harness import OracleSession, ProductSession, close, max_abs
from libbuild import ensure_built
from paged_decode_attention_store_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_built()


DEV = "cuda:0"


def _workload(dtype, Hq, Hkv, D, P, lengths, num_pages, seed, layers=1, window=0):
    order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
    return wl.Workload("test", dtype, Hq, Hkv, D, P, layers, num_pages, order, list(lengths),
                       window=window, scale=1.0 / math.sqrt(D))


# ---------------------------------------------------------------------------
def test_generator_identical_on_cpu_and_gpu(kb):
    k1, v1 = wl.kv_rows(5, 3, [0, 7, 255], [0, 9, 16000], 8, 128)
    k2, v2 = wl.kv_rows(5, 3, [0, 7, 255], [0, 9, 16000], 8, 128, device=DEV)
    assert torch.equal(k1, k2.cpu()) and torch.equal(v1, v2.cpu())
    q1 = wl.q_rows(5, 2, 31, [1, 2], 64, 128, dtype=torch.float32)
    q2 = wl.q_rows(5, 2, 31, [1, 2], 64, 128, dtype=torch.float32, device=DEV)
    assert torch.equal(q1, q2.cpu())


@pytest.mark.parametrize("dtype,Hkv,D", [("bf16", 8, 128), ("f32", 2, 16), ("bf16", 1, 64)])
def test_store_cache_bit_exact(kb, dtype, Hkv, D):
    """Every slot of the written layer equals the oracle's SlotStore after
    the same store_cache (mini-sglang part 4: row i at slot out_loc[i]);
    slots never written stay zero, other layers are untouched."""
    import oracle.attention as OA

    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    P, pages, layers = 16, 40, 3
    kv = torch.zeros((2, layers, pages, P, Hkv, D), dtype=tdt, device=DEV)
    pool = kb.Pool(kv, P, kb.KVP_BF16 if dtype == "bf16" else kb.KVP_F32)
    R = random.Random(1)
    slots = R.sample(range(pages * P), 300)
    k, v = wl.kv_rows(1, 1, 0, list(range(300)), Hkv, D, dtype=tdt, device=DEV)
    kb.store_cache(pool, 1, k, v, torch.tensor(slots, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert kb.kvp_sync_error(pool) == 0
    store = OA.SlotStore()
    kc, vc = wl.kv_rows(1, 1, 0, list(range(300)), Hkv, D, dtype=tdt)
    store.store_cache(slots, kc.double().numpy(), vc.double().numpy())
    gotK = kv[0, 1].reshape(pages * P, Hkv, D).double().cpu().numpy()
    gotV = kv[1, 1].reshape(pages * P, Hkv, D).double().cpu().numpy()
    for sl in range(pages * P):
        if sl in store.k:
            assert np.array_equal(gotK[sl], store.k[sl]) and np.array_equal(gotV[sl], store.v[sl]), f"slot {sl}"
        else:
            assert not gotK[sl].any() and not gotV[sl].any(), f"slot {sl} was written"
    assert not kv[:, 0].any() and not kv[:, 2].any()  # other layers untouched


def test_store_cache_bad_slot_is_flagged_and_skipped(kb):
    P, pages = 4, 8
    kv = torch.zeros((2, 1, pages, P, 2, 16), dtype=torch.float32, device=DEV)
    pool = kb.Pool(kv, P, kb.KVP_F32)
    k, v = wl.kv_rows(2, 0, 0, [0, 1, 2], 2, 16, dtype=torch.float32, device=DEV)
    kb.store_cache(pool, 0, k, v, torch.tensor([3, pages * P, -1], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert kb.kvp_sync_error(pool) == kb.KVP_ERR_BAD_INDEX
    assert kb.kvp_sync_error(pool) == 0  # cleared
    want = torch.zeros_like(kv)
    want[0, 0].view(-1, 2, 16)[3] = k[0]
    want[1, 0].view(-1, 2, 16)[3] = v[0]
    assert torch.equal(kv, want)  # only the valid row was written


@pytest.mark.parametrize("P", [1, 4, 16])
def test_page_table_write_block_and_raw(kb, P):
    """Host bookkeeping's writes land as the oracle's block rows (expand 1)
    and as its token-expanded rows (expand P)."""
    from oracle.pagetable import PageTable

    R = random.Random(P)
    n_pages = 200
    order = list(range(n_pages))
    R.shuffle(order)
    host = kb.HostPageTable(n_pages, P, 4, order)
    opt = PageTable(n_pages, P, free_order=order)
    cols_block = 64
    blk = torch.full((4, cols_block), -1, dtype=torch.int32, device=DEV)
    raw = torch.zeros((5, cols_block * P), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def apply(writes):
        if writes:
            r, c, v = (torch.tensor(x, dtype=torch.int32, device=DEV) for x in zip(*writes))
            kb.page_table_write(blk, r, c, v, 1, err)
            kb.page_table_write(raw, r, c, v, P, err)

    for rid in range(4):
        host.new(rid)
        opt.new(rid)
    for step in range(60):
        rids = [R.randrange(4) for _ in range(R.randrange(1, 6))]
        _, writes, _ = host.append(rids)
        for r in rids:
            opt.append(r)
        apply(writes)
        if step % 7 == 3:
            rid = R.randrange(4)
            k = R.randrange(0, opt.length[rid] + 1)
            apply(host.trim(rid, k))
            opt.trim(rid, k)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for rid in range(4):
        row = opt.block_row(rid)
        assert blk[rid, :len(row)].tolist() == row
        assert raw[rid, :len(row) * P].tolist() == opt.raw_row(rid)
    # an out-of-table write is flagged and skipped
    kb.page_table_write(blk, *(torch.tensor([x], dtype=torch.int32, device=DEV) for x in (9, 0, 1)), 1, err)
    torch.cuda.synchronize()
    assert int(err.item()) == kb.KVP_ERR_BAD_INDEX


def test_copy_pages_bit_exact(kb):
    """copy_pages equals the oracle's whole-page copy (chapter 15, "The
    model": a shared tail page is copied before a private write) on every
    layer, K and V."""
    import oracle.attention as OA

    P, pages, layers, Hkv, D = 16, 12, 2, 8, 128
    kv = torch.randn((2, layers, pages, P, Hkv, D), device=DEV).to(torch.bfloat16)
    stores = []
    for layer in range(layers):  # the oracle's view of the pool, every slot written
        st = OA.SlotStore()
        st.store_cache(list(range(pages * P)), kv[0, layer].reshape(-1, Hkv, D).double().cpu().numpy(),
                       kv[1, layer].reshape(-1, Hkv, D).double().cpu().numpy())
        stores.append(st)
    pool = kb.Pool(kv, P, kb.KVP_BF16)
    src, dst = [1, 5, 7], [2, 9, 0]
    kb.copy_pages(pool, torch.tensor(src, dtype=torch.int32, device=DEV), torch.tensor(dst, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert kb.kvp_sync_error(pool) == 0
    for st in stores:
        for s_, d_ in zip(src, dst):
            st.copy_page(s_, d_, P)
    for layer, st in enumerate(stores):
        gotK = kv[0, layer].reshape(-1, Hkv, D).double().cpu().numpy()
        gotV = kv[1, layer].reshape(-1, Hkv, D).double().cpu().numpy()
        for sl in range(pages * P):
            assert np.array_equal(gotK[sl], st.k[sl]) and np.array_equal(gotV[sl], st.v[sl]), f"layer {layer} slot {sl}"


# ---------------------------------------------------------------------------
# The tiny workload: fp32, 2/2 heads, head_dim 16, page 4, 64 pages, 4
# requests decoding 32 tokens from empty, windows none / 8 / 4.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("W", [None, 8, 4])
def test_tiny_decode_parity(kb, W):
    w = wl.tiny(seed=0, window=W)
    B = 4
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=16)
    orc = OracleSession(w, B)
    for b in range(B):
        prod.new(b)
        orc.new(b)
    window = 0 if W is None else W
    pages_seen = []
    for L in range(1, 33):
        rids = list(range(B))
        pos = [L - 1] * B
        s_gpu = prod.append(rids, pos)
        s_orc = orc.append(rids, pos)
        assert s_gpu == s_orc
        out = prod.attend(0, rids, [L] * B, window, step=L).cpu().numpy()
        slots = prod.gather(rids, [L] * B, window, 40).cpu().numpy()
        tab = prod.table.cpu().numpy()
        for b in range(B):
            ref = orc.attend(0, b, L, window, step=L)
            assert max_abs(out[b], ref) <= 1e-5, f"step {L} request {b}"
            lo = 0 if not window else max(0, L - window)
            want = orc.slots(b, lo, L)
            assert slots[b, :len(want)].tolist() == want and (slots[b, len(want):] == -1).all()
            row = orc.table_row(b)
            assert tab[b, :len(row)].tolist() == row
        if W is not None:
            for b in range(B):
                prod.trim(b, max(0, L + 1 - W))
                orc.trim(b, max(0, L + 1 - W))
        pages_seen.append(prod.host.used())
        assert prod.host.used() == orc.pt.used()
    assert prod.error() == 0
    # per request, the chapter's page counts (4 requests share the pool)
    per_req = {None: 8, 8: 2, 4: 1}[W]
    assert pages_seen[-1] == B * per_req


# ---------------------------------------------------------------------------
# bf16 on the tensor-core kernel (head_dim 128).
# ---------------------------------------------------------------------------
BF16_CASES = [
    # Hq, Hkv, P, lengths, window
    (32, 8, 16, [1, 15, 16, 17, 250, 1000, 3001], 0),   # GQA 4, ragged and split requests
    (64, 8, 16, [3, 700, 2100], 0),                       # GQA 8
    (8, 8, 16, [129, 2000], 0),                           # no grouping
    (64, 4, 16, [33, 1500], 0),                           # GQA 16 (two MMA column tiles)
    (16, 2, 8, [5, 800, 64], 0),                          # 2 KV heads, page 8
    (32, 16, 16, [90, 1200], 0),                          # 16 KV heads: two head groups
    (32, 8, 16, [1000, 37, 2500], 100),                   # window without trim
    (32, 8, 1, [300, 1, 77], 0),                          # page size 1
    # GQA 8 keeps one Q buffer: runs of one-stage pieces reuse it back to back
    (64, 8, 8, [7, 8, 300, 1, 2, 3, 9, 1, 1, 17, 4, 33, 2, 5], 0),
]


@pytest.mark.parametrize("case", range(len(BF16_CASES)))
def test_bf16_block_decode_parity(kb, case):
    Hq, Hkv, P, lengths, window = BF16_CASES[case]
    B = len(lengths)
    steps = 3
    num_pages = sum(-(-(L + steps) // P) for L in lengths) + 8
    w = _workload("bf16", Hq, Hkv, 128, P, lengths, num_pages, seed=100 + case)
    cols = max(-(-(L + steps) // P) for L in lengths) + 2
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=cols, seed=case)
    orc = OracleSession(w, B, seed=case)
    for b, L in enumerate(lengths):
        prod.new(b)
        orc.new(b)
        assert prod.append([b] * L, list(range(L))) == orc.append([b] * L, list(range(L)))
    lens = list(lengths)
    for step in range(1, steps + 1):
        rids = list(range(B))
        assert prod.append(rids, lens) == orc.append(rids, lens)
        lens = [L + 1 for L in lens]
        out = prod.attend(0, rids, lens, window, step=step).float().cpu().numpy()
        for b in range(B):
            ref = orc.attend(0, b, lens[b], window, step=step)
            close(out[b], ref, "bf16", f"step {step} request {b} (L={lens[b]})")
    tab = prod.table.cpu().numpy()
    for b in range(B):
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    assert prod.error() == 0


@pytest.mark.parametrize("P,mode", [(16, "block"), (4, "block"), (32, "block"), (1, "raw"), (8, "raw")])
def test_bf16_mixed_contiguous_and_scattered_groups(kb, P, mode):
    """Pages handed out mostly in address order, with a few swapped, so that
    some 16-token groups are 16 contiguous, 16-aligned slots, some are
    contiguous but misaligned and some are scattered; two layers, so that both
    layers' K and V are addressed. Every kind of group must give the same
    result as the oracle."""
    lengths = [700, 45, 1290, 16, 333]
    B, layers, steps = len(lengths), 2, 2
    num_pages = sum(-(-(L + steps) // P) for L in lengths) + 8
    order = list(range(num_pages))
    rng = random.Random(P)
    for _ in range(max(2, num_pages // 40)):
        i, j = rng.randrange(num_pages), rng.randrange(num_pages)
        order[i], order[j] = order[j], order[i]
    w = wl.Workload("test", "bf16", 32, 8, 128, P, layers, num_pages, wl.free_stack_for_order(order),
                    list(lengths), scale=1.0 / math.sqrt(128))
    cols = (max(lengths) + steps + 64) if mode == "raw" else max(-(-(L + steps) // P) for L in lengths) + 2
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=cols, mode=mode, seed=11)
    orc = OracleSession(w, B, mode=mode, seed=11, raw_cols=prod.table.shape[1] if mode == "raw" else None)
    for b, L in enumerate(lengths):
        prod.new(b)
        orc.new(b)
        assert prod.append([b] * L, list(range(L))) == orc.append([b] * L, list(range(L)))
    lens = list(lengths)
    for step in range(1, steps + 1):
        rids = list(range(B))
        assert prod.append(rids, lens) == orc.append(rids, lens)
        lens = [L + 1 for L in lens]
        for layer in range(layers):
            out = prod.attend(layer, rids, lens, 0, step=step).float().cpu().numpy()
            for b in range(B):
                close(out[b], orc.attend(layer, b, lens[b], 0, step=step), "bf16", f"layer {layer} step {step} request {b}")
    assert prod.error() == 0


@pytest.mark.parametrize("P", [16, 1])
def test_bf16_raw_location_parity_with_dummy_row(kb, P):
    """mini-sglang layout: (2, layers, pages + 1 dummy, P, 8, 128), raw token
    locations, a dummy row pointing into the dummy page, 2 layers."""
    lengths = [1, 33, 900, 1500, 2047]
    B, layers, steps = len(lengths), 2, 2
    num_pages = sum(-(-(L + steps) // P) for L in lengths) + 4
    w = _workload("bf16", 64, 8, 128, P, lengths, num_pages, seed=7 + P, layers=layers)
    max_seq = 4096
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=max_seq, mode="raw", seed=3)
    orc = OracleSession(w, B, mode="raw", seed=3, raw_cols=max_seq)
    assert prod.table.shape[1] == orc.raw.page_table.shape[1]
    for b, L in enumerate(lengths):
        prod.new(b)
        orc.new(b)
        assert prod.append([b] * L, list(range(L))) == orc.append([b] * L, list(range(L)))
    # the dummy request (row B) writes one row into the dummy page
    dummy_slot = num_pages * P
    for layer in range(layers):
        k, v = wl.kv_rows(3, layer, B, 0, 8, 128, dtype=torch.bfloat16, device=DEV)
        kb.store_cache(prod.pool, layer, k, v, torch.tensor([dummy_slot], dtype=torch.int32, device=DEV))
        kc, vc = wl.kv_rows(3, layer, B, 0, 8, 128, dtype=torch.bfloat16)
        orc.stores[layer].store_cache([dummy_slot], kc.float().numpy(), vc.float().numpy())
    lens = list(lengths)
    for step in range(1, steps + 1):
        rids = list(range(B))
        assert prod.append(rids, lens) == orc.append(rids, lens)
        lens = [L + 1 for L in lens]
        for layer in range(layers):
            out = prod.attend(layer, rids + [B], lens + [1], 0, step=step).float().cpu().numpy()
            for b in range(B):
                close(out[b], orc.attend(layer, b, lens[b], 0, step=step), "bf16", f"layer {layer} request {b}")
            # one attended row: the output is that row's value, per KV head
            vd = wl.kv_rows(3, layer, B, 0, 8, 128, dtype=torch.bfloat16)[1][0].float().numpy()
            assert max_abs(out[B], np.repeat(vd, 8, axis=0)) <= 1e-2
    tab = prod.table.cpu().numpy()
    for b in range(B):
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    assert (tab[B] == num_pages * P).all()
    assert prod.error() == 0


def test_sliding_window_with_front_holes(kb):
    """Window 64, page 16: history built by the real append + trim path, so
    released pages are reused and the table has -1 holes at the front."""
    W, P = 64, 16
    lengths = [500, 70, 1]
    B, steps = len(lengths), 20
    num_pages = B * (-(-(W - 1) // P) + 2) + 4
    w = _workload("bf16", 32, 8, 128, P, lengths, num_pages, seed=21, window=W)
    cols = (max(lengths) + steps) // P + 2
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=cols, seed=9)
    orc = OracleSession(w, B, seed=9)
    for b, L in enumerate(lengths):
        prod.new(b)
        orc.new(b)
        for t in range(L):
            assert prod.append([b], [t]) == orc.append([b], [t])
            prod.trim(b, max(0, t + 2 - W))
            orc.trim(b, max(0, t + 2 - W))
    lens = list(lengths)
    for step in range(1, steps + 1):
        rids = list(range(B))
        assert prod.append(rids, lens) == orc.append(rids, lens)
        lens = [L + 1 for L in lens]
        out = prod.attend(0, rids, lens, W, step=step).float().cpu().numpy()
        for b in range(B):
            close(out[b], orc.attend(0, b, lens[b], W, step=step), "bf16", f"step {step} request {b}")
        for b in range(B):
            prod.trim(b, max(0, lens[b] + 1 - W))
            orc.trim(b, max(0, lens[b] + 1 - W))
        assert prod.host.used() == orc.pt.used() <= B * (-(-(W - 1) // P) + 1)
    tab = prod.table.cpu().numpy()
    assert (tab[0, :10] == -1).all()  # released front pages
    for b in range(B):
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    assert prod.error() == 0


def test_prefix_sharing_copy_on_write(kb):
    """2 prompts of 50 tokens (page 16: the shared tail page holds 2 rows),
    3 forks each; every fork's first append copies the tail page."""
    P, prompt = 16, 50
    suffix = [5, 17, 40, 1, 16, 33]
    num_pages = 2 * 4 + sum(-(-(prompt + s + 3) // P) - prompt // P for s in suffix) + 4
    w = _workload("bf16", 32, 8, 128, P, [0] * 8, num_pages, seed=31)
    prod = ProductSession(kb, w, DEV, max_requests=8, cols=8, seed=4)
    orc = OracleSession(w, 8, seed=4)
    for base in (6, 7):
        prod.new(base)
        orc.new(base)
        assert prod.append([base] * prompt, list(range(prompt))) == orc.append([base] * prompt, list(range(prompt)))
    for f in range(6):
        prod.fork(6 + f // 3, f)
        orc.fork(6 + f // 3, f)
    # first suffix token of every fork while the prompt requests still hold the tail
    assert prod.append(list(range(6)), [prompt] * 6) == orc.append(list(range(6)), [prompt] * 6)
    assert prod.n_copies == 6
    for base in (6, 7):
        prod.release(base)
        orc.release(base)
    lens = [prompt + 1] * 6
    for f in range(6):
        n = suffix[f] - 1
        if n > 0:
            pos = list(range(lens[f], lens[f] + n))
            assert prod.append([f] * n, pos) == orc.append([f] * n, pos)
            lens[f] += n
    for step in range(1, 4):
        rids = list(range(6))
        assert prod.append(rids, lens) == orc.append(rids, lens)
        lens = [L + 1 for L in lens]
        out = prod.attend(0, rids, lens, 0, step=step).float().cpu().numpy()
        for b in range(6):
            close(out[b], orc.attend(0, b, lens[b], 0, step=step), "bf16", f"step {step} request {b}")
    assert prod.host.refcounts() == orc.pt.ref
    assert prod.error() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_device_detected_errors_leave_the_context_usable(kb, dtype):
    D = 128 if dtype == "bf16" else 16
    Hq, Hkv, P = (32, 8, 16) if dtype == "bf16" else (2, 2, 4)
    lengths = [40, 100]
    num_pages = 20 if P == 16 else 64
    w = _workload(dtype, Hq, Hkv, D, P, lengths, num_pages, seed=41)
    prod = ProductSession(kb, w, DEV, max_requests=2, cols=40, seed=5)
    for b, L in enumerate(lengths):
        prod.new(b)
        prod.append([b] * L, list(range(L)))
    assert prod.error() == 0
    # a hole inside the attended range
    saved = prod.table.clone()
    prod.table[1, 2] = -1
    out = prod.attend(0, [0, 1], lengths, 0, step=1)
    torch.cuda.synchronize()
    assert prod.error() == kb.KVP_ERR_BAD_INDEX
    assert torch.isfinite(out.float()).all()
    prod.table.copy_(saved)
    # a length beyond the table's capacity and a zero length
    for bad in (40 * P + 1, 0):
        out = prod.attend(0, [0, 1], [lengths[0], bad], 0, step=1)
        torch.cuda.synchronize()
        assert prod.error() == kb.KVP_ERR_BAD_INDEX
        assert not out[1].float().any()
    # the context is still usable and correct afterwards
    orc = OracleSession(w, 2, seed=5)
    for b, L in enumerate(lengths):
        orc.new(b)
        orc.append([b] * L, list(range(L)))
    out = prod.attend(0, [0, 1], lengths, 0, step=2).float().cpu().numpy()
    for b in range(2):
        close(out[b], orc.attend(0, b, lengths[b], 0, step=2), dtype, f"request {b}")
    assert prod.error() == 0
