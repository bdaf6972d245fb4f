"""store_cache_and_attention (one launch per layer) against the three calls
it replaces: page_table_write, store_cache, paged_decode_attention.

Two identical sessions step the same requests; one issues the separate
calls, the other the fused one (with the step's new-page table writes on
the first layer). Outputs, tables and the whole K/V buffer must be
bit-identical, and the outputs must match the oracle (bf16: 2e-2).
"""

import math

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
    # dtype, Hq, Hkv, D, P, mode, lengths
    ("bf16", 32, 8, 128, 16, "block", [15, 16, 17, 31, 700, 1, 2047]),  # steps cross page boundaries
    ("bf16", 64, 8, 128, 8, "block", [7, 8, 300]),
    ("bf16", 32, 8, 128, 16, "raw", [15, 33, 900]),
    ("bf16", 16, 2, 128, 1, "raw", [1, 5, 400]),  # every position a new page
    ("f32", 4, 2, 16, 4, "block", [3, 4, 9]),     # no fused kernel: the three calls in sequence
]


def _i32(xs):
    return torch.tensor(list(xs), dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_step_equals_the_separate_calls(kb, case):
    dtype, Hq, Hkv, D, P, mode, lengths = CASES[case]
    B, layers, steps = len(lengths), 2, 20
    num_pages = sum(-(-(L + steps) // P) for L in lengths) + 8
    order = wl.free_stack_for_order(wl.permutation(40 + case, num_pages))
    w = wl.Workload("fused", dtype, Hq, Hkv, D, P, layers, num_pages, order, list(lengths),
                    scale=1.0 / math.sqrt(D))
    if mode == "raw":
        cols = max(lengths) + steps + 32
    else:
        cols = max(-(-(L + steps) // P) for L in lengths) + 2
    sep = ProductSession(kb, w, DEV, max_requests=B, cols=cols, mode=mode, seed=4)
    fus = ProductSession(kb, w, DEV, max_requests=B, cols=cols, mode=mode, seed=4)
    orc = OracleSession(w, B, mode=mode, seed=4, raw_cols=sep.table.shape[1] if mode == "raw" else None)
    for b, L in enumerate(lengths):
        for s in (sep, fus):
            s.new(b)
            s.append([b] * L, list(range(L)))
        orc.new(b)
        orc.append([b] * L, list(range(L)))
    tmode = kb.KVP_RAW_LOCATIONS if mode == "raw" else kb.KVP_BLOCK_TABLE
    rids = list(range(B))
    lens = list(lengths)
    ws = kb.alloc_workspace(fus.pool, B, Hq, device=DEV)
    for step in range(1, steps + 1):
        # separate calls
        slots_sep = sep.append(rids, lens)
        # fused: host bookkeeping, then one launch per layer
        slots, writes, cows = fus.host.append(rids)
        assert slots == slots_sep and not cows
        orc.append(rids, lens)
        new_lens = [L + 1 for L in lens]
        out_loc, lens_t = _i32(slots), _i32(new_lens)
        tw = None
        if writes:
            r, c, v = zip(*writes)
            tw = (_i32(r), _i32(c), _i32(v))
        for layer in range(layers):
            q = wl.q_rows(4, step, layer, rids, Hq, D, dtype=fus.dt, device=DEV)
            k, v = wl.kv_rows(4, layer, rids, lens, Hkv, D, dtype=fus.dt, device=DEV)
            out_f = torch.empty_like(q)
            kb.store_cache_and_attention(fus.pool, layer, q, k, v, out_loc, fus.table, tmode, lens_t, 0, w.scale,
                                         out_f, ws, table_rows=_i32(rids), table_writes=tw if layer == 0 else None)
            out_s = sep.attend(layer, rids, new_lens, 0, step=step)
            assert torch.equal(out_f, out_s), f"step {step} layer {layer}: fused output differs"
            if step % 5 == 0:
                got = out_f.float().cpu().numpy()
                for b in rids:
                    close(got[b], orc.attend(layer, b, new_lens[b], 0, step=step), dtype,
                          f"step {step} layer {layer} request {b}")
        lens = new_lens
    torch.cuda.synchronize()
    assert torch.equal(fus.table, sep.table), "tables differ"
    assert torch.equal(fus.kv, sep.kv), "K/V buffers differ"
    assert fus.error() == 0 and sep.error() == 0
