"""Pins of the oracle's rewind(n) and multi-token verify attention (CPU only).

rewind(n): "Week 3 Day 3: Paged KV Cache" (tiny-llm) adds a hook that drops
the newest n logical tokens, frees the whole pages no longer needed and
shortens the valid length of the last page. Anchors: a shadow model with
rewinds between appends, forks, trims and releases (every row read back
through the table, reference counts equal to the table entries, no leaks);
the exact page count after a rewind; rewind followed by re-appending the
same number of tokens rebuilds the same table; three planted mutants.

Multi-token verify (speculative decoding, which the same page names as the
user of rewind): the M newest tokens are queries at once, query j attending
what a single-token step with context L - M + j + 1 attends. Anchors: the
chapter-15 decode loop run step by step over the same rows and queries, and
PyTorch's scaled_dot_product_attention in float64 with an explicit mask.
"""

import math
import random

import numpy as np
import pytest
import torch

import oracle.attention as A
import oracle.decode as Dm
from oracle.pagetable import OutOfPages, PageTable
from paged_decode_attention_store_gb300 import workloads as wl


# ---------------------------------------------------------------------------
# rewind
# ---------------------------------------------------------------------------
def _invariants(pt, shadow):
    P = []
    cnt = [0] * len(pt.ref)
    for tb in pt.table.values():
        for p in tb:
            cnt[p] += 1
    if cnt != list(pt.ref):
        P.append("reference counts differ from the block-table entries")
    if len(set(pt.free)) != len(pt.free) or any(pt.ref[p] != 0 for p in pt.free):
        P.append("free list holds a page twice or a referenced page")
    if len(pt.free) + sum(1 for r in pt.ref if r > 0) != len(pt.ref):
        P.append("a page is neither free nor referenced")
    for rid, rows in shadow.items():
        lo = pt.dropped[rid] * pt.page
        if pt.length[rid] != len(rows):
            P.append(f"length of request {rid}")
        elif pt.rows(rid, lo, len(rows)) != rows[lo:]:
            P.append(f"rows of request {rid} differ from the shadow")
        elif len(pt.table[rid]) != -(-len(rows) // pt.page) - pt.dropped[rid]:
            P.append(f"request {rid} holds {len(pt.table[rid])} pages for {len(rows)} rows")
    return P


def check_rewind_shadow(PT, seed, n_ops=500, n_pages=24, page=4, max_live=5):
    R = random.Random(seed)
    pt = PT(n_pages, page)
    shadow = {}
    nxt = ctr = 0
    for step in range(n_ops):
        op = R.choice(["append"] * 5 + ["rewind"] * 2 + ["new", "fork", "trim", "release"])
        ids = list(shadow)
        try:
            if op == "new" and len(ids) < max_live:
                pt.new(nxt); shadow[nxt] = []; nxt += 1
            elif op == "append" and ids:
                rid = R.choice(ids)
                for _ in range(R.randrange(1, 7)):
                    ctr += 1
                    pt.append(rid, (ctr, -ctr))
                    shadow[rid].append((ctr, -ctr))
            elif op == "rewind" and ids:
                rid = R.choice(ids)
                floor = pt.dropped[rid] * page if pt.dropped[rid] else 0
                n = R.randrange(0, len(shadow[rid]) - floor + 1)
                pt.rewind(rid, n)
                del shadow[rid][len(shadow[rid]) - n:]
            elif op == "fork" and ids and len(ids) < max_live:
                s = R.choice(ids); pt.fork(s, nxt); shadow[nxt] = list(shadow[s]); nxt += 1
            elif op == "trim" and ids:
                rid = R.choice(ids); pt.trim(rid, R.randrange(0, len(shadow[rid]) + 1))
            elif op == "release" and ids:
                rid = R.choice(ids); pt.release(rid); del shadow[rid]
        except OutOfPages:
            pass
        P = _invariants(pt, shadow)
        if P:
            return [f"seed {seed} op {step} ({op}): {p}" for p in P[:3]]
    for rid in list(shadow):
        pt.release(rid)
    if len(pt.free) != n_pages or any(pt.ref):
        return [f"seed {seed}: pages leaked after releasing every request"]
    return []


def check_rewind_restores_layout(PT):
    """Rewind then re-append as many tokens: the same pages in the same order."""
    P = []
    for page, L, n in ((4, 14, 6), (4, 16, 8), (1, 9, 9), (16, 40, 25), (3, 10, 1)):
        pt = PT(32, page)
        pt.new(0)
        pt.new(1)
        for i in range(L):
            pt.append(0, i)
        pt.append(1, "x")
        before = (pt.block_row(0), list(pt.free), list(pt.ref))
        gone = pt.rewind(0, n)
        want_gone = -(-L // page) - -(-(L - n) // page)
        if len(gone) != want_gone:
            P.append(f"page {page}: rewinding {n} of {L} freed {len(gone)} pages, not {want_gone}")
        for i in range(n):
            pt.append(0, ("again", i))
        if (pt.block_row(0), list(pt.free), list(pt.ref)) != before:
            P.append(f"page {page}: re-appending after rewind({n}) did not rebuild the table")
    return P


def check_rewind_limits(PT):
    P = []
    pt = PT(16, 4)
    pt.new(0)
    for i in range(13):
        pt.append(0, i)
    pt.trim(0, 9)  # pages 0 and 1 released
    for bad in (6, 14, -1):  # into the released front, past the start, negative
        try:
            pt.rewind(0, bad)
            P.append(f"rewind({bad}) was accepted")
        except ValueError:
            pass
    if pt.length[0] != 13:
        P.append("a refused rewind changed the length")
    pt.rewind(0, 5)  # down to 8 rows: exactly the released front
    if pt.length[0] != 8 or pt.table[0] != [] or pt.rows(0, 8, 8) != []:
        P.append("rewinding to the released front left pages or rows")
    return P


def all_rewind_problems(PT=PageTable):
    P = check_rewind_restores_layout(PT) + check_rewind_limits(PT)
    for seed in range(8):
        P += check_rewind_shadow(PT, seed)
    P += check_rewind_shadow(PT, 99, n_pages=64, page=3, max_live=8)
    return P


def test_rewind_pins():
    assert all_rewind_problems() == []


class LeakyRewind(PageTable):
    def rewind(self, rid, n):
        L = self.length[rid]
        self.length[rid] = L - n
        keep = -(-(L - n) // self.page) - self.dropped[rid]
        del self.table[rid][keep:]  # pages dropped from the table but never returned
        return []


class RewindOneTooMany(PageTable):
    def rewind(self, rid, n):
        gone = super().rewind(rid, n)
        if self.table[rid] and n and self.length[rid] % self.page:
            self._unref(self.table[rid].pop())
        return gone


class RewindKeepsPages(PageTable):
    def rewind(self, rid, n):
        self.length[rid] -= n
        return []


@pytest.mark.parametrize("mutant", [LeakyRewind, RewindOneTooMany, RewindKeepsPages], ids=lambda m: m.__name__)
def test_rewind_mutant_is_caught(mutant):
    try:
        problems = all_rewind_problems(mutant)
    except (IndexError, ValueError) as e:
        problems = [repr(e)]
    assert problems, f"{mutant.__name__} survived"


# ---------------------------------------------------------------------------
# multi-token verify attention
# ---------------------------------------------------------------------------
VERIFY_CASES = ((None, 0, 4, 4), (6, 0, 4, 3), (6, 2, 2, 4), (9, 3, 4, 5), (None, 0, 1, 1), (5, 1, 1, 2))
# (W, S, page, M)


def _verify_oracle(W, S, page, M, L0=13, seed=7, Hq=4, Hkv=2, D=16):
    """Append L0 + M rows (no trim), then the verify outputs of the M newest."""
    pt = PageTable(64, page, free_order=wl.free_stack_for_order(wl.permutation(seed, 64)))
    pt.new(0)
    store = A.SlotStore()
    L = L0 + M
    k, v = wl.kv_rows(seed, 0, 0, list(range(L)), Hkv, D, dtype=torch.float32)
    slots = [pt.append(0)["slot"] for _ in range(L)]
    store.store_cache(slots, k.numpy(), v.numpy())
    row = pt.block_row(0)
    outs = []
    for j, pos in enumerate(A.verify_positions(L, M, W, S)):
        q = wl.q_rows(seed, j + 1, 0, [0], Hq, D, dtype=torch.float32)[0].numpy()
        sl = [s for p in pos for s in A.gather_block(row, page, p, p + 1)]
        outs.append(A.attend_request(store, q, sl, 1.0 / math.sqrt(D)))
    return np.stack(outs), k.numpy(), v.numpy()


def check_verify_equals_decode_loop():
    """Query j of a verify equals decode step j of chapter 15's loop (append
    one token, attend, trim) run over the same rows and queries."""
    P = []
    for W, S, page, M in VERIFY_CASES:
        L0, seed, Hq, Hkv, D = 13, 7, 4, 2, 16
        got, k, v = _verify_oracle(W, S, page, M, L0, seed, Hq, Hkv, D)
        pt = PageTable(64, page, free_order=wl.free_stack_for_order(wl.permutation(seed, 64)))
        pt.new(0)
        dec = Dm.BlockDecoder(pt, W, 1.0 / math.sqrt(D), sinks=S)
        dec.prefill(0, k[:L0], v[:L0])
        for j in range(M):
            q = wl.q_rows(seed, j + 1, 0, [0], Hq, D, dtype=torch.float32).numpy()
            _, _, out = dec.step([0], q, k[L0 + j:L0 + j + 1], v[L0 + j:L0 + j + 1])
            if np.max(np.abs(out[0] - got[j])) > 1e-12:
                P.append(f"W={W} S={S} page={page} M={M}: query {j} differs from decode step {j}")
                break
    return P


def check_verify_library_sdpa():
    """Against torch SDPA (float64) with the causal window mask written out."""
    P = []
    for W, S, page, M in VERIFY_CASES:
        L0, seed, Hq, Hkv, D = 13, 7, 4, 2, 16
        got, k, v = _verify_oracle(W, S, page, M, L0, seed, Hq, Hkv, D)
        L = L0 + M
        mask = torch.zeros((M, L), dtype=torch.bool)
        for j in range(M):
            p = L - M + j  # the query's own position
            for t in range(p + 1):
                in_window = W is None or t >= p + 1 - (W - S)
                mask[j, t] = in_window or t < S
        q = torch.stack([wl.q_rows(seed, j + 1, 0, [0], Hq, D, dtype=torch.float64)[0] for j in range(M)])
        qt = q.permute(1, 0, 2)[None]  # [1, Hq, M, D]
        kt = torch.as_tensor(k, dtype=torch.float64).permute(1, 0, 2)[None]
        vt = torch.as_tensor(v, dtype=torch.float64).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=1.0 / math.sqrt(D),
                                                               enable_gqa=True)[0].permute(1, 0, 2).numpy()
        if np.max(np.abs(ref - got)) > 1e-12:
            P.append(f"W={W} S={S} page={page} M={M}: differs from masked SDPA")
    return P


def test_verify_equals_the_decode_loop():
    assert check_verify_equals_decode_loop() == []


def test_verify_equals_masked_sdpa():
    assert check_verify_library_sdpa() == []


def test_whole_sequence_prefill_equals_causal_sdpa():
    """A chunk that is the whole sequence (L0 = 0: every token a query) is
    textbook causal attention: torch SDPA with its own is_causal mask
    (float64, GQA), no mask written here."""
    for page, M in ((4, 21), (1, 7), (16, 40)):
        Hq, Hkv, D, seed = 4, 2, 16, 11
        got, k, v = _verify_oracle(None, 0, page, M, L0=0, seed=seed, Hq=Hq, Hkv=Hkv, D=D)
        q = torch.stack([wl.q_rows(seed, j + 1, 0, [0], Hq, D, dtype=torch.float64)[0] for j in range(M)])
        qt = q.permute(1, 0, 2)[None]
        kt = torch.as_tensor(k, dtype=torch.float64).permute(1, 0, 2)[None]
        vt = torch.as_tensor(v, dtype=torch.float64).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=1.0 / math.sqrt(D),
                                                               enable_gqa=True)[0].permute(1, 0, 2).numpy()
        assert np.max(np.abs(ref - got)) <= 1e-12, f"page {page}, {M} tokens"


def test_verify_positions_readings():
    # context 10, 3 verify tokens, no window: causal prefixes
    assert A.verify_positions(10, 3, None) == [list(range(8)), list(range(9)), list(range(10))]
    # window 4, 1 sink
    assert A.verify_positions(10, 2, 4, 1) == [[0, 6, 7, 8], [0, 7, 8, 9]]
    with pytest.raises(ValueError):
        A.verify_positions(3, 4, None)


@pytest.mark.parametrize("name", ["query sees its successor", "window not shifted per query"])
def test_verify_mutant_is_caught(name, monkeypatch):
    orig = A.verify_positions
    if name == "query sees its successor":
        monkeypatch.setattr(A, "verify_positions", lambda L, M, W, S=0: [
            A.attended_positions(min(L, L - M + j + 2), W, S) for j in range(M)])
    else:
        monkeypatch.setattr(A, "verify_positions", lambda L, M, W, S=0: [
            sorted(set(orig(L, M, W, S)[0]) | {L - M + j}) for j in range(M)])
    assert check_verify_equals_decode_loop() + check_verify_library_sdpa()
