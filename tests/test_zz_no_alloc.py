"""paged_decode_attention_noalloc: attention for callers that cannot allocate.

Some callers cannot allocate device memory where they run attention (inside
another framework's memory pool, under a budget that forbids new
reservations, plug-in hosts that receive only their buffers). This entry
point takes its split-K scratch from a fixed array inside the library, so
such a caller passes only inputs and outputs. It must return what
paged_decode_attention returns with a caller-provided workspace, on
consecutive calls that reuse the array. The file is collected last so that a
run stopping at the first failure has already run every other test.
"""

import math

import pytest
import torch

from gpu_harness import ProductSession, max_abs
from libbuild import ensure_built
from paged_decode_attention_store_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def kb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_built()


@pytest.mark.parametrize("Hq,Hkv,lengths", [(32, 8, [3000, 17, 1200, 640]), (64, 8, [1, 2500, 700])])
def test_noalloc_matches_the_workspace_entry_point(kb, Hq, Hkv, lengths):
    P, D, seed = 16, 128, 61
    steps = 2
    num_pages = sum(-(-(L + steps) // P) for L in lengths) + 4
    order = wl.free_stack_for_order(wl.permutation(seed, num_pages))
    w = wl.Workload("noalloc", "bf16", Hq, Hkv, D, P, 1, num_pages, order, list(lengths), scale=1.0 / math.sqrt(D))
    B = len(lengths)
    prod = ProductSession(kb, w, DEV, max_requests=B, cols=max(-(-(L + steps) // P) for L in lengths) + 1, seed=seed)
    for b, L in enumerate(lengths):
        prod.new(b)
        prod.append([b] * L, list(range(L)))
    lens = list(lengths)
    rids = list(range(B))
    for step in range(1, steps + 1):  # two calls in a row, each after one more decode token
        prod.append(rids, lens)
        lens = [L + 1 for L in lens]
        want = prod.attend(0, rids, lens, 0, step=step)
        q = wl.q_rows(seed, step, 0, rids, Hq, D, dtype=torch.bfloat16, device=DEV)
        got = torch.empty_like(q)
        kb.paged_decode_attention_noalloc(prod.pool, 0, q, prod.table, kb.KVP_BLOCK_TABLE,
                                          torch.tensor(lens, dtype=torch.int32, device=DEV), 0, w.scale, got,
                                          table_rows=torch.tensor(rids, dtype=torch.int32, device=DEV))
        torch.cuda.synchronize()
        assert max_abs(got.float().cpu().numpy(), want.float().cpu().numpy()) <= 2e-2, f"step {step}"
    assert prod.error() == 0
