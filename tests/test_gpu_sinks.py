"""Attention-sink windows on the GPU against the oracle.

Chapter 15 of silicon_compiler_from_scratch ("A Paged KV Cache and
Sliding-Window Attention"), exercise "Attention sinks": a windowed step
keeps the first S rows and the last W - S. Requests are built through the
real append + trim path (the trim keeps the sink pages), then decode steps
run with the separate calls and with the fused one-launch step. Slots read
(gather_indices), tables and page counts are bit-exact against the oracle;
outputs within 2e-2 (bf16) or 1e-5 (fp32); fused and separate outputs
bit-identical.
"""

import math

import numpy as np
import pytest
import torch

from gpu_harness import OracleSession, ProductSession, close
from libbuild import ensure_built
from paged_decode_attention_store_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def kb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_built()


CASES = [
    # dtype, Hq, Hkv, D, P, mode, W, S, lengths
    ("bf16", 32, 8, 128, 16, "block", 100, 2, [1, 50, 99, 100, 101, 300, 1000]),
    ("bf16", 32, 8, 128, 4, "block", 64, 4, [3, 63, 64, 65, 500]),
    ("bf16", 64, 8, 128, 16, "raw", 200, 2, [10, 250, 1200]),
    ("bf16", 16, 2, 128, 1, "raw", 40, 3, [5, 41, 90]),
    ("bf16", 32, 8, 128, 16, "block", 4096, 2, [4000, 4100, 9000]),  # the bench's window, sinks spanning one stage
    ("f32", 4, 2, 16, 4, "block", 12, 2, [3, 12, 13, 40]),
]


def _setup(kb, case, seed):
    dtype, Hq, Hkv, D, P, mode, W, S, lengths = CASES[case]
    B, steps = len(lengths), 12
    per_req = -(-S // P) + -(-(W - S) // P) + 2
    num_pages = B * per_req + -(-16 // P) + 8  # room for one prefill chunk before its trim
    order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
    w = wl.Workload("sinks", dtype, Hq, Hkv, D, P, 1, num_pages, order, list(lengths), window=W,
                    scale=1.0 / math.sqrt(D))
    mx = max(lengths) + steps
    cols = mx + 32 if mode == "raw" else -(-mx // P) + 2
    if mode == "raw":  # the raw-location table is no wider than the pool has tokens
        num_pages = max(num_pages, -(-cols // P))
        order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
        w = wl.Workload("sinks", dtype, Hq, Hkv, D, P, 1, num_pages, order, list(lengths), window=W,
                        scale=1.0 / math.sqrt(D))
    return w, B, steps, cols


def _prefill(sessions, orc, lengths, W, S):
    """History through the real path: every row appended, then trimmed to what
    the first decode step can read (keep_from = L + 1 - (W - S))."""
    for b, L in enumerate(lengths):
        for s in sessions:
            s.new(b)
        orc.new(b)
        t = 0
        while t < L:
            n = min(16, L - t)
            for s in sessions:
                s.append([b] * n, list(range(t, t + n)))
                s.trim(b, max(0, t + n + 1 - (W - S)), sinks=S)
            orc.append([b] * n, list(range(t, t + n)))
            orc.trim(b, max(0, t + n + 1 - (W - S)), sinks=S)
            t += n


@pytest.mark.parametrize("case", range(len(CASES)))
def test_sink_decode_parity(kb, case):
    dtype, Hq, Hkv, D, P, mode, W, S, lengths = CASES[case]
    w, B, steps, cols = _setup(kb, case, 60 + case)
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=cols, mode=mode, seed=5)
    orc = OracleSession(w, B, mode=mode, seed=5, raw_from_pages=True)
    _prefill([prod], orc, lengths, W, S)
    assert prod.host.used() == orc.pt.used()
    lens = list(lengths)
    rids = list(range(B))
    for step in range(1, steps + 1):
        assert prod.append(rids, lens) == orc.append(rids, lens)
        lens = [L + 1 for L in lens]
        out = prod.attend(0, rids, lens, W, step=step, sinks=S).float().cpu().numpy()
        got = prod.gather(rids, lens, W, W, sinks=S).cpu().numpy()
        for b in rids:
            want = orc.span_slots(b, lens[b], W, S)
            assert len(want) == min(lens[b], W)
            assert got[b, :len(want)].tolist() == want and (got[b, len(want):] == -1).all()
            close(out[b], orc.attend(0, b, lens[b], W, step=step, sinks=S), dtype, f"step {step} request {b} (L={lens[b]})")
        for b in rids:
            prod.trim(b, max(0, lens[b] + 1 - (W - S)), sinks=S)
            orc.trim(b, max(0, lens[b] + 1 - (W - S)), sinks=S)
        assert prod.host.used() == orc.pt.used()
    tab = prod.table.cpu().numpy()
    for b in rids:
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    assert prod.error() == 0


@pytest.mark.parametrize("case", [0, 2, 3, 4])
def test_sink_fused_step_equals_separate_calls(kb, case):
    dtype, Hq, Hkv, D, P, mode, W, S, lengths = CASES[case]
    w, B, steps, cols = _setup(kb, case, 80 + case)
    sep = ProductSession(kb, w, DEV, max_requests=B, cols=cols, mode=mode, seed=6)
    fus = ProductSession(kb, w, DEV, max_requests=B, cols=cols, mode=mode, seed=6)
    orc = OracleSession(w, B, mode=mode, seed=6, raw_from_pages=True)
    _prefill([sep, fus], orc, lengths, W, S)
    tmode = kb.KVP_RAW_LOCATIONS if mode == "raw" else kb.KVP_BLOCK_TABLE
    rids = list(range(B))
    lens = list(lengths)
    ws = kb.alloc_workspace(fus.pool, B, Hq, device=DEV)
    i32 = lambda xs: torch.tensor(list(xs), dtype=torch.int32, device=DEV)  # noqa: E731
    for step in range(1, steps + 1):
        slots_sep = sep.append(rids, lens)
        slots, writes, cows = fus.host.append(rids)
        assert slots == slots_sep and not cows
        orc.append(rids, lens)
        new_lens = [L + 1 for L in lens]
        tw = tuple(i32(x) for x in zip(*writes)) if writes else None
        q = wl.q_rows(6, step, 0, rids, Hq, D, dtype=fus.dt, device=DEV)
        k, v = wl.kv_rows(6, 0, rids, lens, Hkv, D, dtype=fus.dt, device=DEV)
        out_f = torch.empty_like(q)
        kb.store_cache_and_attention(fus.pool, 0, q, k, v, i32(slots), fus.table, tmode, i32(new_lens), W, w.scale,
                                     out_f, ws, table_rows=i32(rids), table_writes=tw, sinks=S)
        out_s = sep.attend(0, rids, new_lens, W, step=step, sinks=S)
        assert torch.equal(out_f, out_s), f"step {step}: fused output differs"
        got = out_f.float().cpu().numpy()
        for b in rids:
            close(got[b], orc.attend(0, b, new_lens[b], W, step=step, sinks=S), dtype, f"step {step} request {b}")
        for b in rids:
            kf = max(0, new_lens[b] + 1 - (W - S))
            sep.trim(b, kf, sinks=S)
            fus.trim(b, kf, sinks=S)
            orc.trim(b, kf, sinks=S)
        lens = new_lens
    torch.cuda.synchronize()
    assert torch.equal(fus.table, sep.table) and torch.equal(fus.kv, sep.kv)
    assert fus.error() == 0 and sep.error() == 0


def test_sink_arguments_are_checked(kb):
    w, B, steps, cols = _setup(kb, 0, 1)
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=cols, seed=1)
    prod.new(0)
    prod.append([0] * 5, list(range(5)))
    for W, S in ((8, 8), (8, 9), (8, -1)):
        with pytest.raises(kb.KvpError):
            prod.attend(0, [0], [5], W, step=1, sinks=S)
    # without a window the sinks change nothing
    a = prod.attend(0, [0], [5], 0, step=1, sinks=3)
    b = prod.attend(0, [0], [5], 0, step=1)
    assert torch.equal(a, b)
