"""paged_decode_attention_noalloc: attention for callers that cannot allocate.

Some callers cannot allocate device memory where they run attention (inside
another framework's memory pool, under a budget that forbids new
reservations, plug-in hosts that receive only their buffers). This entry
point takes its split-K scratch from a fixed array inside the library, so
such a caller passes only inputs and outputs.

Both entry points launch the same kernels on the same inputs and differ only
in where the partials live, so their outputs must be bit-identical, on
consecutive calls that reuse the array; each output is also checked against
the oracle. A shape whose scratch does not fit the array must be refused
before anything runs. The file is collected last so that a run stopping at
the first failure has already run every other test.
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
    # dtype, Hq, Hkv, D, P, lengths, window, sinks
    ("bf16", 32, 8, 128, 16, [3000, 17, 1200, 640], 0, 0),  # tensor-core kernel, split requests
    ("bf16", 64, 8, 128, 16, [1, 2500, 700], 0, 0),
    ("bf16", 32, 8, 128, 16, [5000, 300, 2100], 1024, 2),    # window with attention sinks
    ("f32", 4, 2, 64, 4, [300, 9, 77], 0, 0),                # general kernel
    ("f32", 4, 2, 64, 4, [300, 9, 77], 40, 0),
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,P,lengths,window,sinks", CASES)
def test_noalloc_matches_the_workspace_entry_point(kb, dtype, Hq, Hkv, D, P, lengths, window, sinks):
    seed, steps = 61, 2
    num_pages = sum(-(-(L + steps) // P) for L in lengths) + 4
    order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
    w = wl.Workload("noalloc", dtype, Hq, Hkv, D, P, 1, num_pages, order, list(lengths), scale=1.0 / math.sqrt(D))
    B = len(lengths)
    cols = max(-(-(L + steps) // P) for L in lengths) + 1
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=cols, seed=seed)
    orc = OracleSession(w, max_requests=B, seed=seed)
    for b, L in enumerate(lengths):
        for s in (prod, orc):
            s.new(b)
            s.append([b] * L, list(range(L)))
    lens = list(lengths)
    rids = list(range(B))
    for step in range(1, steps + 1):  # two calls in a row, each after one more decode token
        for s in (prod, orc):
            s.append(rids, lens)
        lens = [L + 1 for L in lens]
        want = prod.attend(0, rids, lens, window, step=step, sinks=sinks)
        q = wl.q_rows(seed, step, 0, rids, Hq, D, dtype=prod.dt, device=DEV)
        got = torch.full_like(q, float("nan"))
        kb.paged_decode_attention_noalloc(prod.pool, 0, q, prod.table, kb.KVP_BLOCK_TABLE,
                                          torch.tensor(lens, dtype=torch.int32, device=DEV), window, w.scale, got,
                                          table_rows=torch.tensor(rids, dtype=torch.int32, device=DEV), sinks=sinks)
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"step {step}: outputs differ from the workspace entry point"
        g = got.float().cpu().numpy()
        for b in rids:
            ref = orc.attend(0, b, lens[b], window, step, sinks=sinks)
            close(g[b], ref, dtype, f"step {step} request {b}")
        if window > 0:
            for b in rids:
                for s in (prod, orc):
                    s.trim(b, max(0, lens[b] + 1 - (window - sinks)), sinks=sinks)
    assert prod.error() == 0


def test_noalloc_refuses_a_shape_larger_than_its_array(kb):
    """128 query heads on one KV head need more split-K scratch than the
    fixed array holds: the call is refused on the host and nothing is
    written."""
    D, P, Hq, Hkv, B = 128, 16, 128, 1, 2
    pool_kv = torch.zeros((2, 1, 8, P, Hkv, D), dtype=torch.bfloat16, device=DEV)
    pool = kb.Pool(pool_kv, P, kb.KVP_BF16)
    assert kb.paged_decode_attention_workspace_size(pool, B, Hq) > 12 << 20
    table = torch.arange(B * 4, dtype=torch.int32, device=DEV).view(B, 4)
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device=DEV)
    out = torch.full_like(q, 7.0)
    with pytest.raises(kb.KvpError) as e:
        kb.paged_decode_attention_noalloc(pool, 0, q, table, kb.KVP_BLOCK_TABLE,
                                          torch.tensor([5, 9], dtype=torch.int32, device=DEV), 0, 1.0, out)
    assert e.value.code == kb.KVP_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a refused call wrote its output"
    assert kb.kvp_sync_error(pool) == 0
