"""Speculative decoding on the GPU: multi-token verify attention and rewind.

Each step appends M drafted tokens per request (host bookkeeping, table
writes, store_cache), verifies them with paged_verify_attention (query j at
position L - M + j, causal, same window and sinks as a decode step), accepts
a random number of them and rewinds the rest (kvp_host_rewind: whole pages
past the new length go back, tail first), then trims for the next step.
Against the oracle: slots, tables and page counts bit-exact; every query's
output within 2e-2 (bf16) or 1e-5 (fp32).
"""

import math
import random

import pytest
import torch

import oracle.attention as OA
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
    # dtype, Hq, Hkv, D, P, mode, M, W, S, lengths
    ("bf16", 32, 8, 128, 16, "block", 4, 0, 0, [1, 15, 16, 300, 1000, 2047]),  # 16 columns per KV head
    ("bf16", 64, 8, 128, 16, "block", 4, 0, 0, [5, 700, 1500]),                # 32 columns: two warps per KV head
    ("bf16", 64, 8, 128, 16, "block", 8, 0, 0, [9, 400]),                      # 64 columns: four warps per KV head
    ("bf16", 32, 8, 128, 16, "block", 2, 100, 2, [3, 99, 150, 600]),           # window with sinks
    ("bf16", 32, 8, 128, 1, "raw", 3, 0, 0, [4, 33, 500]),                     # every position its own page
    ("bf16", 16, 2, 128, 8, "raw", 5, 64, 0, [6, 64, 300]),
    ("f32", 4, 2, 16, 4, "block", 3, 12, 2, [3, 12, 40]),                      # general kernel
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_speculative_steps_match_the_oracle(kb, case):
    dtype, Hq, Hkv, D, P, mode, M, W, S, lengths = CASES[case]
    B, steps = len(lengths), 10
    mx = max(lengths) + steps * M + M
    num_pages = sum(-(-(L + steps * M + M) // P) for L in lengths) + 16
    if mode == "raw":
        num_pages = max(num_pages, -(-(mx + 32) // P))
    order = wl.free_stack_for_order(wl.permutation(90 + case, num_pages))
    w = wl.Workload("verify", dtype, Hq, Hkv, D, P, 1, num_pages, order, list(lengths), window=W, sinks=S,
                    scale=1.0 / math.sqrt(D))
    cols = mx + 32 if mode == "raw" else -(-mx // P) + 2
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=cols, mode=mode, seed=12)
    orc = OracleSession(w, B, mode=mode, seed=12, raw_from_pages=True)
    for b, L in enumerate(lengths):
        prod.new(b)
        orc.new(b)
        assert prod.append([b] * L, list(range(L))) == orc.append([b] * L, list(range(L)))
        if W:
            prod.trim(b, max(0, L + 1 - (W - S)), sinks=S)
            orc.trim(b, max(0, L + 1 - (W - S)), sinks=S)
    tmode = kb.KVP_RAW_LOCATIONS if mode == "raw" else kb.KVP_BLOCK_TABLE
    ws = kb.alloc_verify_workspace(prod.pool, B, M, Hq, device=DEV)
    R = random.Random(case)
    rids = list(range(B))
    lens = list(lengths)
    i32 = lambda xs: torch.tensor(list(xs), dtype=torch.int32, device=DEV)  # noqa: E731
    for step in range(1, steps + 1):
        # M drafted tokens per request, stored before the verify
        rr = [b for b in rids for _ in range(M)]
        pp = [lens[b] + j for b in rids for j in range(M)]
        assert prod.append(rr, pp) == orc.append(rr, pp)
        ctx = [L + M for L in lens]
        q = torch.stack([wl.q_rows(12, step * 64 + j, 0, rids, Hq, D, dtype=prod.dt, device=DEV) for j in range(M)],
                        dim=1).contiguous()
        out = torch.empty_like(q)
        kb.paged_verify_attention(prod.pool, 0, q, prod.table, tmode, i32(ctx), W, w.scale, out, ws,
                                  table_rows=i32(rids), sinks=S)
        got = out.float().cpu().numpy()
        for b in rids:
            for j, pos in enumerate(OA.verify_positions(ctx[b], M, W, S)):
                qj = q[b, j].float().cpu().numpy()
                sl = [s for p in pos for s in orc.slots(b, p, p + 1)]
                ref = OA.attend_request(orc.stores[0], qj, sl, w.scale)
                close(got[b, j], ref, dtype, f"step {step} request {b} query {j} (L={ctx[b]})")
        # accept a random number of drafts, rewind the rest, trim for the next step
        for b in rids:
            acc = R.randrange(0, M + 1)
            gone = prod.host.rewind(b, M - acc)
            prod._write(gone)
            assert [c for _, c, _ in gone] == orc.pt.rewind(b, M - acc)
            lens[b] += acc
            if W:
                prod.trim(b, max(0, lens[b] + 1 - (W - S)), sinks=S)
                orc.trim(b, max(0, lens[b] + 1 - (W - S)), sinks=S)
        assert prod.host.used() == orc.pt.used()
        assert [prod.host.length(b)[0] for b in rids] == lens
    tab = prod.table.cpu().numpy()
    for b in rids:
        row = orc.table_row(b)
        assert tab[b, :len(row)].tolist() == row
    assert prod.error() == 0


def test_single_token_verify_equals_decode(kb):
    Hq, Hkv, D, P = 32, 8, 128, 16
    lengths = [1, 17, 300, 2049, 640]
    B = len(lengths)
    num_pages = sum(-(-L // P) for L in lengths) + 8
    order = wl.free_stack_for_order(wl.permutation(5, num_pages))
    w = wl.Workload("v1", "bf16", Hq, Hkv, D, P, 1, num_pages, order, lengths, scale=1.0 / math.sqrt(D))
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=-(-max(lengths) // P) + 1, seed=3)
    for b, L in enumerate(lengths):
        prod.new(b)
        prod.append([b] * L, list(range(L)))
    for W, S in ((0, 0), (200, 3)):
        a = prod.attend(0, list(range(B)), lengths, W, step=1, sinks=S)
        q = wl.q_rows(3, 1, 0, list(range(B)), Hq, D, dtype=torch.bfloat16, device=DEV)
        out = torch.empty((B, 1, Hq, D), dtype=torch.bfloat16, device=DEV)
        ws = kb.alloc_verify_workspace(prod.pool, B, 1, Hq, device=DEV)
        i32 = lambda xs: torch.tensor(list(xs), dtype=torch.int32, device=DEV)  # noqa: E731
        kb.paged_verify_attention(prod.pool, 0, q[:, None].contiguous(), prod.table, kb.KVP_BLOCK_TABLE,
                                  i32(lengths), W, w.scale, out, ws, table_rows=i32(range(B)), sinks=S)
        assert torch.equal(out[:, 0], a)
    assert prod.error() == 0


def test_verify_arguments_are_checked(kb):
    Hq, Hkv, D, P = 32, 8, 128, 16
    w = wl.Workload("v2", "bf16", Hq, Hkv, D, P, 1, 8, list(range(8)), [3], scale=0.1)
    prod = ProductSession(kb, w, DEV, max_requests=1, cols=4, seed=3)
    prod.new(0)
    prod.append([0] * 3, [0, 1, 2])
    i32 = lambda xs: torch.tensor(list(xs), dtype=torch.int32, device=DEV)  # noqa: E731
    q = torch.zeros((1, 33, Hq, D), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(kb.KvpError):  # more than 32 query tokens
        kb.paged_verify_attention(prod.pool, 0, q, prod.table, kb.KVP_BLOCK_TABLE, i32([3]), 0, 0.1,
                                  torch.empty_like(q), kb.alloc_verify_workspace(prod.pool, 1, 1, Hq, device=DEV))
    # more query tokens than the context holds: flagged on the device, output zero
    q = torch.ones((1, 4, Hq, D), dtype=torch.bfloat16, device=DEV)
    out = torch.ones_like(q)
    kb.paged_verify_attention(prod.pool, 0, q, prod.table, kb.KVP_BLOCK_TABLE, i32([3]), 0, 0.1, out,
                              kb.alloc_verify_workspace(prod.pool, 1, 4, Hq, device=DEV))
    torch.cuda.synchronize()
    assert prod.error() == kb.KVP_ERR_BAD_INDEX
    assert not out.any()
