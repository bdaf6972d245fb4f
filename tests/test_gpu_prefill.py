"""Chunked prefill (paged_prefill_attention) against the oracle.

Requests hold a prefix in the pages; a chunk of new tokens is appended
through the host bookkeeping and stored, then attended at once: query j at
position L - q_len + j attends causally what a one-token step with that
context would (oracle: verify_positions, the decode formula per query).
bf16 pools with head_dim 128 run on the tcgen05 tensor cores (tiles of 128
query rows = 128 / G tokens x G heads, 128-key blocks), fp32 on the general
kernel. Every written row within 2e-2 (bf16) or 1e-5 (fp32); rows past a
request's chunk are left untouched.
"""

import math

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
    # dtype, Hq, Hkv, D, P, mode, chunk, prefixes, q_lens, W, S
    ("bf16", 32, 8, 128, 16, "block", 300, [0, 100, 1000, 17], [300, 300, 50, 1], 0, 0),  # 32 tokens per tile
    ("bf16", 64, 8, 128, 16, "block", 128, [0, 500], [128, 77], 0, 0),                    # GQA 8: 16 tokens per tile
    ("bf16", 8, 8, 128, 1, "raw", 200, [333, 0], [200, 129], 0, 0),                       # no grouping, scattered slots
    ("bf16", 32, 8, 128, 16, "block", 256, [700, 40], [256, 256], 200, 2),                # window with sinks
    ("bf16", 64, 4, 128, 4, "block", 64, [90, 3], [64, 40], 0, 0),                        # GQA 16, page 4
    ("f32", 4, 2, 16, 4, "block", 20, [5, 30], [20, 7], 12, 2),                           # general kernel
    ("bf16", 32, 8, 128, 16, "raw", 200, [500, 33], [200, 150], 0, 0),                    # raw table, page 16 (TMA)
    ("bf16", 32, 8, 128, 16, "block", 300, [1000, 0], [300, 300], 128, 0),                # window, no sinks
    ("bf16", 16, 8, 128, 16, "block", 96, [70, 0], [96, 5], 0, 0),                        # GQA 2: 64 tokens per tile
    ("bf16", 32, 8, 128, 32, "block", 200, [300, 45], [200, 190], 0, 0),                  # page 32: two groups a page
    ("bf16", 32, 8, 128, 64, "block", 160, [1000, 7], [160, 160], 256, 16),               # page 64, a whole sink group
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill_chunk_matches_the_oracle(kb, case):
    dtype, Hq, Hkv, D, P, mode, C, prefixes, q_lens, W, S = CASES[case]
    B = len(prefixes)
    lens = [p + q for p, q in zip(prefixes, q_lens)]
    num_pages = sum(-(-L // P) for L in lens) + 8
    if mode == "raw":
        num_pages = max(num_pages, -(-(max(lens) + 32) // P))
    order = wl.free_stack_for_order(wl.permutation(120 + case, num_pages))
    w = wl.Workload("prefill", dtype, Hq, Hkv, D, P, 1, num_pages, order, prefixes, window=W, sinks=S,
                    scale=1.0 / math.sqrt(D))
    cols = max(lens) + 32 if mode == "raw" else -(-max(lens) // P) + 2
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=cols, mode=mode, seed=8)
    orc = OracleSession(w, B, mode=mode, seed=8, raw_from_pages=True)
    for b in range(B):
        prod.new(b)
        orc.new(b)
        n = lens[b]  # prefix and chunk rows, stored through the same path
        assert prod.append([b] * n, list(range(n))) == orc.append([b] * n, list(range(n)))
    i32 = lambda xs: torch.tensor(list(xs), dtype=torch.int32, device=DEV)  # noqa: E731
    q = torch.stack([wl.q_rows(8, 500 + j, 0, list(range(B)), Hq, D, dtype=prod.dt, device=DEV) for j in range(C)],
                    dim=1).contiguous()
    out = torch.full_like(q, 7.0)
    tmode = kb.KVP_RAW_LOCATIONS if mode == "raw" else kb.KVP_BLOCK_TABLE
    kb.paged_prefill_attention(prod.pool, 0, q, prod.table, tmode, i32(lens), W, w.scale, out, q_lens=i32(q_lens),
                               table_rows=i32(range(B)), sinks=S)
    torch.cuda.synchronize()
    assert prod.error() == 0
    got = out.float().cpu().numpy()
    for b in range(B):
        for j, pos in enumerate(OA.verify_positions(lens[b], q_lens[b], W if W else None, S)):
            sl = [s for p in pos for s in orc.slots(b, p, p + 1)]
            ref = OA.attend_request(orc.stores[0], q[b, j].float().cpu().numpy(), sl, w.scale)
            close(got[b, j], ref, dtype, f"request {b} query {j} (L={lens[b]}, q_len={q_lens[b]})")
        assert (got[b, q_lens[b]:] == 7.0).all(), f"request {b}: rows past the chunk were written"


def test_prefill_single_token_equals_decode(kb):
    """A one-token chunk is a decode step: equal to paged_decode_attention
    within the bf16 rounding of the two kernels' accumulation orders."""
    Hq, Hkv, D, P = 32, 8, 128, 16
    lengths = [1, 17, 300, 2049]
    B = len(lengths)
    num_pages = sum(-(-L // P) for L in lengths) + 8
    order = wl.free_stack_for_order(wl.permutation(9, num_pages))
    w = wl.Workload("p1", "bf16", Hq, Hkv, D, P, 1, num_pages, order, lengths, scale=1.0 / math.sqrt(D))
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=-(-max(lengths) // P) + 1, seed=3)
    for b, L in enumerate(lengths):
        prod.new(b)
        prod.append([b] * L, list(range(L)))
    i32 = lambda xs: torch.tensor(list(xs), dtype=torch.int32, device=DEV)  # noqa: E731
    dec = prod.attend(0, list(range(B)), lengths, 0, step=1)
    q = wl.q_rows(3, 1, 0, list(range(B)), Hq, D, dtype=torch.bfloat16, device=DEV)[:, None].contiguous()
    out = torch.empty_like(q)
    kb.paged_prefill_attention(prod.pool, 0, q, prod.table, kb.KVP_BLOCK_TABLE, i32(lengths), 0, w.scale, out,
                               table_rows=i32(range(B)))
    torch.cuda.synchronize()
    assert (out[:, 0].float() - dec.float()).abs().max().item() <= 2e-2
    assert prod.error() == 0


def test_prefill_bad_lengths_zero_the_request(kb):
    """A request whose chunk is longer than its context records
    KVP_ERR_BAD_INDEX and gets zero rows; the other request is unaffected."""
    Hq, Hkv, D, P, C = 32, 8, 128, 16, 128
    lens, q_lens = [300, 40], [128, 64]
    B = len(lens)
    num_pages = sum(-(-L // P) for L in lens) + 8
    order = wl.free_stack_for_order(wl.permutation(77, num_pages))
    w = wl.Workload("pbad", "bf16", Hq, Hkv, D, P, 1, num_pages, order, [0, 0], scale=1.0 / math.sqrt(D))
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=-(-max(lens) // P) + 2, seed=5)
    orc = OracleSession(w, B, seed=5)
    for b in range(B):
        prod.new(b)
        orc.new(b)
        assert prod.append([b] * lens[b], list(range(lens[b]))) == orc.append([b] * lens[b], list(range(lens[b])))
    i32 = lambda xs: torch.tensor(list(xs), dtype=torch.int32, device=DEV)  # noqa: E731
    q = torch.stack([wl.q_rows(9, 700 + j, 0, list(range(B)), Hq, D, dtype=prod.dt, device=DEV) for j in range(C)],
                    dim=1).contiguous()
    out = torch.full_like(q, 7.0)
    kb.paged_prefill_attention(prod.pool, 0, q, prod.table, kb.KVP_BLOCK_TABLE, i32(lens), 0, w.scale, out,
                               q_lens=i32(q_lens), table_rows=i32(range(B)))
    torch.cuda.synchronize()
    assert prod.error() == kb.KVP_ERR_BAD_INDEX
    assert (out[1] == 0).all(), "the invalid request's rows are not zero"
    got = out.float().cpu().numpy()
    for j, pos in enumerate(OA.verify_positions(lens[0], q_lens[0], None, 0)):
        sl = [s_ for p_ in pos for s_ in orc.slots(0, p_, p_ + 1)]
        ref = OA.attend_request(orc.stores[0], q[0, j].float().cpu().numpy(), sl, w.scale)
        close(got[0, j], ref, "bf16", f"query {j}")
