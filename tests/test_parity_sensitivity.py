"""The GPU parity bounds are tight enough to see a lost page, row or stage.

Chapter 15's "Mutation tests" makes the point that a loose tolerance or a
bound-only check hides conservative errors. These CPU tests plant the
mistake a kernel could make at a piece boundary (one 16-row page, one row
or one 16-row stage left out of a request's attended rows, or read twice) in
the ORACLE's input and check that the result moves by more than the bound
the GPU tests apply, at every context length those tests reach:

- random inputs (``tests/gpu_harness.close``): max |out' - out| must exceed
  REL_K * 2^-8 * max |out| for a dropped page at every length, and for a
  dropped row up to 4,096 rows;
- coded inputs (``tests/test_gpu_coded``): some entry of a zero query head
  must move by more than that test's bound for it (1.25 * 2^-8 of itself,
  + 2^-20) for a dropped or doubled row or stage at every length, up to the
  16,128 rows of the longest raw-table context.
"""

import numpy as np
import pytest

import oracle.attention as OA
from gpu_harness import REL_K
from test_gpu_coded import ABS, REL_ZERO_Q
from paged_decode_attention_store_gb300 import workloads as wl

LENGTHS = [512, 2500, 3001, 4096, 9000, 16128]


def _rows(inputs, L, Hkv=8, D=128, rid=3):
    k, v = inputs.kv_rows(0, 0, rid, list(range(L)), Hkv, D)
    return k.double().numpy(), v.double().numpy()


def _q(inputs, Hq, D=128, rid=3):
    return inputs.q_rows(0, 1, 0, [rid], Hq, D)[0].double().numpy()


@pytest.mark.parametrize("L", LENGTHS)
@pytest.mark.parametrize("Hq", [32, 64])
def test_random_input_bound_sees_a_dropped_page(L, Hq):
    K, V = _rows(wl, L)
    q = _q(wl, Hq)
    scale = 1.0 / np.sqrt(128)
    ref = OA.decode_attention(q, K, V, scale)
    gate = REL_K * 2.0 ** -8 * np.abs(ref).max()
    p0 = (L // 2) // 16 * 16  # a page in the middle, where a split would cut
    keep = np.r_[0:p0, p0 + 16:L]
    moved = np.abs(OA.decode_attention(q, K[keep], V[keep], scale) - ref).max()
    assert moved > gate, f"L={L}: a dropped page moves the output by {moved}, bound {gate}"
    if L <= 4096:
        keep = np.r_[0:p0 + 5, p0 + 6:L]
        moved = np.abs(OA.decode_attention(q, K[keep], V[keep], scale) - ref).max()
        assert moved > gate, f"L={L}: a dropped row moves the output by {moved}, bound {gate}"


def _coded_bound_fails(ref, got):
    """Whether the coded test's bound for the zero query heads rejects ``got``."""
    r, g = ref[0::2], got[0::2]
    return bool((np.abs(g - r) > REL_ZERO_Q * np.abs(r) + ABS).any())


@pytest.mark.parametrize("L", LENGTHS)
def test_coded_bound_sees_a_lost_or_doubled_row_or_stage(L):
    inputs = wl.CodedInputs()
    K, V = _rows(inputs, L)
    q = _q(inputs, 64)
    scale = 1.0 / np.sqrt(128)
    ref = OA.decode_attention(q, K, V, scale)
    p0 = (L // 3) // 16 * 16
    cases = {
        "dropped row": np.r_[0:p0 + 7, p0 + 8:L],
        "doubled row": np.r_[0:p0 + 8, p0 + 7:L],
        "dropped stage": np.r_[0:p0, p0 + 16:L],
        "doubled stage": np.r_[0:p0 + 16, p0:L],
        "stage read from the next one": np.r_[0:p0, p0 + 16:p0 + 32, p0 + 16:L],
    }
    for what, idx in cases.items():
        got = OA.decode_attention(q, K[idx], V[idx], scale)
        assert _coded_bound_fails(ref, got), f"L={L}: {what} stays within the coded bound"
