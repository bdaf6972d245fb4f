"""Pins of the oracle's dense decode attention and its decode loop (CPU only).

Independent anchors: closed forms (one row, equal scores, two rows),
invariances that hold for softmax attention, PyTorch's library
scaled_dot_product_attention in float64 (a special case the oracle reduces
to), and the chapter-15 window checks (a window at least as long as the
context changes nothing; a short one changes the result; the windowed step
equals a recomputation over exactly the last W tokens, regenerated from the
input generator rather than read back from the cache).
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as A
import oracle.decode as Dm
from oracle.pagetable import PageTable
from paged_decode_attention_store_gb300 import workloads as wl


def _rand(shape, seed):
    return np.random.RandomState(seed).standard_normal(shape)


def _sdpa(q, K, V, scale):
    """Library reference: q [Hq, D], K/V [n, Hkv, D] -> [Hq, D] (float64)."""
    qt = torch.as_tensor(q, dtype=torch.float64)[None, :, None, :]
    kt = torch.as_tensor(K, dtype=torch.float64).permute(1, 0, 2)[None]
    vt = torch.as_tensor(V, dtype=torch.float64).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale, enable_gqa=True)
    return o[0, :, 0, :].numpy()


# ---------------------------------------------------------------------------
def check_closed_forms():
    P = []
    q, k, v = _rand(16, 1), _rand((1, 16), 2), _rand((1, 16), 3)
    if not np.array_equal(A.attention_one(q, k, v, 0.25), v[0]):
        P.append("one row: output is not that row's value")
    V = _rand((7, 16), 4)
    if not np.allclose(A.attention_one(np.zeros(16), _rand((7, 16), 5), V, 0.25), V.mean(0), atol=1e-14):
        P.append("equal scores: output is not the mean of the values")
    K2, V2, q2, sc = _rand((2, 8), 6), _rand((2, 8), 7), _rand(8, 8), 0.3
    s0, s1 = sc * K2[0] @ q2, sc * K2[1] @ q2
    sig = 1.0 / (1.0 + math.exp(-(s1 - s0)))
    if not np.allclose(A.attention_one(q2, K2, V2, sc), V2[0] + sig * (V2[1] - V2[0]), atol=1e-14):
        P.append("two rows: output differs from the logistic closed form")
    return P


def check_library_sdpa():
    P = []
    for Hq, Hkv, n, D, seed in ((8, 2, 37, 16, 1), (4, 4, 5, 8, 2), (32, 8, 130, 128, 3), (6, 1, 1, 4, 4)):
        q, K, V = _rand((Hq, D), seed), _rand((n, Hkv, D), seed + 10), _rand((n, Hkv, D), seed + 20)
        sc = 1.0 / math.sqrt(D)
        got = A.decode_attention(q, K, V, sc)
        if not np.allclose(got, _sdpa(q, K, V, sc), atol=1e-12, rtol=0):
            P.append(f"Hq={Hq} Hkv={Hkv} n={n} D={D}: differs from torch SDPA")
    return P


def check_invariances():
    P = []
    q, K, V = _rand(12, 30), _rand((20, 12), 31), _rand((20, 12), 32)
    base = A.attention_one(q, K, V, 0.4)
    shifted = A.attention_one(q, K + 2.5 * q / (q @ q), V, 0.4)  # every score + 0.4 * 2.5
    if not np.allclose(base, shifted, atol=1e-12):
        P.append("a common shift of the scores changed the output")
    perm = np.random.RandomState(33).permutation(20)
    if not np.allclose(base, A.attention_one(q, K[perm], V[perm], 0.4), atol=1e-12):
        P.append("permuting the rows changed the output")
    if np.any(base < V.min(0) - 1e-12) or np.any(base > V.max(0) + 1e-12):
        P.append("output left the convex hull of the values")
    V2 = _rand((20, 12), 34)
    lin = A.attention_one(q, K, 2.0 * V - 3.0 * V2, 0.4)
    if not np.allclose(lin, 2.0 * base - 3.0 * A.attention_one(q, K, V2, 0.4), atol=1e-12):
        P.append("output is not linear in the values")
    return P


def _decode_run(W, steps, P=4, seed=3, Hq=4, Hkv=2, D=16, pt_class=PageTable, sinks=0):
    """Oracle decode of one request; returns per-step (L, lo, q, out, pages in use)."""
    order = wl.free_stack_for_order(wl.permutation(seed, 64))
    pt = pt_class(64, P, free_order=order)
    pt.new(0)
    dec = Dm.BlockDecoder(pt, W, 1.0 / math.sqrt(D), sinks=sinks)
    res = []
    for L in range(1, steps + 1):
        q = wl.q_rows(seed, L, 0, [0], Hq, D, dtype=torch.float32).numpy()
        k, v = wl.kv_rows(seed, 0, [0], [L - 1], Hkv, D, dtype=torch.float32)
        _, _, out = dec.step([0], q, k.numpy(), v.numpy())
        lo = 0 if W is None else L - min(L, W)
        res.append((L, lo, q[0], out[0], pt.used()))
    return res


def check_window_semantics():
    P = []
    Hkv, D = 2, 16
    full = _decode_run(None, 13)
    wide = _decode_run(20, 13)
    for (L, _, _, a, _), (_, _, _, b, _) in zip(full, wide):
        if np.max(np.abs(a - b)) > 1e-12:
            P.append(f"step {L}: a window longer than the context changed the result")
    narrow = _decode_run(3, 13)
    if max(np.max(np.abs(a[3] - b[3])) for a, b in zip(full, narrow)) < 1e-3:
        P.append("a window of 3 made no difference: the window is not applied")
    for W in (2, 3, 5, 8):
        for L, lo, q, out, _ in _decode_run(W, 17):
            k, v = wl.kv_rows(3, 0, 0, list(range(max(0, L - W), L)), Hkv, D, dtype=torch.float32)
            ref = _sdpa(q, k.numpy(), v.numpy(), 1.0 / math.sqrt(D))
            if np.max(np.abs(out - ref)) > 1e-12:
                P.append(f"W={W} step {L}: differs from attention over exactly the last {W} tokens")
                break
    return P


def check_decode_page_counts(pt_class=PageTable):
    """The decode loop keeps exactly the pages the window rule predicts."""
    P = []
    for W, page in ((None, 4), (8, 4), (6, 2), (3, 1)):
        for L, _, _, _, used in _decode_run(W, 24, P=page, pt_class=pt_class):
            kf = 0 if W is None else max(0, L + 1 - W)
            want = -(-L // page) - kf // page
            if used != want:
                P.append(f"W={W} page={page} after step {L}: {used} pages, rule says {want}")
                break
    return P


SINK_CASES = ((6, 2, 4), (8, 2, 2), (5, 1, 1), (8, 4, 4), (9, 3, 2), (7, 2, 8))  # W, S, page


def check_sink_semantics():
    """Chapter 15, exercise "Attention sinks": the first S rows plus the last
    W - S, so the context is still W rows. Each step must equal attention
    over exactly those positions, with K/V regenerated from the generator
    (not read back through the table)."""
    P = []
    Hkv, D = 2, 16
    plain = _decode_run(6, 15)
    zero = _decode_run(6, 15, sinks=0)
    if any(np.max(np.abs(a[3] - b[3])) > 0 for a, b in zip(plain, zero)):
        P.append("zero sinks differ from the plain window")
    for W, S, page in SINK_CASES:
        for L, _, q, out, _ in _decode_run(W, 21, P=page, sinks=S):
            want = list(range(L)) if L <= W else list(range(S)) + list(range(L - (W - S), L))
            if len(want) != min(L, W):
                P.append("the sink context is not W rows")
            k, v = wl.kv_rows(3, 0, 0, want, Hkv, D, dtype=torch.float32)
            ref = _sdpa(q, k.numpy(), v.numpy(), 1.0 / math.sqrt(D))
            if np.max(np.abs(out - ref)) > 1e-12:
                P.append(f"W={W} S={S} page={page} step {L}: differs from the first {S} plus the last {W - S} rows")
                break
    # with sinks the result differs from the plain window once the window has slid
    a, b = _decode_run(6, 12, sinks=2), _decode_run(6, 12)
    if np.max(np.abs(a[-1][3] - b[-1][3])) < 1e-3:
        P.append("sinks made no difference after the window slid")
    return P


def check_sink_page_counts(pt_class=PageTable):
    """Pages in use equal a brute-force count: page j (of the ceil(L/P)
    pages written) is kept iff it holds a row the next step can read, a sink
    row (< S) or a row at or after keep_from = L + 1 - (W - S)."""
    P = []
    for W, S, page in SINK_CASES:
        for L, _, _, _, used in _decode_run(W, 24, P=page, sinks=S, pt_class=pt_class):
            kf = max(0, L + 1 - (W - S))
            need = sum(1 for j in range(-(-L // page))
                       if any(r < S or r >= kf for r in range(j * page, min(L, (j + 1) * page))))
            if used != need:
                P.append(f"W={W} S={S} page={page} after step {L}: {used} pages, brute force says {need}")
                break
    return P


def all_attention_problems():
    return (check_closed_forms() + check_library_sdpa() + check_invariances()
            + check_window_semantics() + check_decode_page_counts() + check_sink_semantics()
            + check_sink_page_counts())


def test_closed_forms():
    assert check_closed_forms() == []


def test_reduces_to_library_sdpa():
    assert check_library_sdpa() == []


def test_invariances():
    assert check_invariances() == []


def test_window_semantics():
    assert check_window_semantics() == []


def test_decode_loop_page_counts():
    assert check_decode_page_counts() == []


def test_sink_semantics():
    assert check_sink_semantics() == []


def test_sink_page_counts():
    assert check_sink_page_counts() == []


def test_sink_positions_and_rows():
    # context 10, window 6, 2 sinks: rows 0, 1 and 6..9
    assert A.attended_positions(10, 6, 2) == [0, 1, 6, 7, 8, 9]
    assert A.attended_positions(6, 6, 2) == list(range(6))
    assert A.attended_positions(7, 6, 2) == [0, 1, 3, 4, 5, 6]
    assert A.attended_positions(10, 6, 0) == list(range(4, 10))
    assert A.attended_positions(10, None, 3) == list(range(10))
    with pytest.raises(ValueError):
        A.sink_window(10, 4, 4)
    # the sink page stays in the table while the window slides past it
    pt = PageTable(16, 4)
    pt.new(0)
    for _ in range(14):
        pt.append(0)
    assert pt.trim(0, 9, sink_rows=2) == [1]
    assert pt.block_row(0)[:3] == [pt.table[0][0], -1, pt.table[0][1]]
    assert pt.slot(0, 1) == pt.table[0][0] * 4 + 1
    with pytest.raises(IndexError):
        pt.slot(0, 5)
    assert pt.trim(0, 12, sink_rows=2) == [2]
    with pytest.raises(ValueError):
        pt.trim(0, 12, sink_rows=5)


def test_reading_a_hole_is_an_error():
    with pytest.raises(IndexError):
        A.gather_block([-1, 3], 4, 2, 6)
    with pytest.raises(IndexError):
        A.gather_raw([-1, 5, 6], 0, 3)
    assert A.gather_block([-1, 3], 4, 4, 6) == [12, 13]


def test_window_lo_readings():
    # No window: everything; W = 1: only the current token; W >= L: everything.
    assert A.window_lo(10, None) == 0 and A.window_lo(10, 0) == 0 and A.window_lo(10, -1) == 0
    assert A.window_lo(10, 1) == 9 and A.window_lo(10, 10) == 0 and A.window_lo(10, 4) == 6


# ---------------------------------------------------------------------------
# Mutation tests: planted mistakes in the oracle's attention and decode loop.
# ---------------------------------------------------------------------------
def _attention_no_scale(q, K, V, scale):
    return _orig_attention_one(q, K, V, 1.0)


def _attention_unnormalised(q, K, V, scale):
    q, K, V = (np.asarray(x, dtype=np.float64) for x in (q, K, V))
    s = scale * (K @ q)
    return np.exp(s - s.max()) @ V


def _decode_attention_kv_swapped(q, K, V, scale):
    return _orig_decode_attention(q, V, K, scale)


def _decode_attention_modulo_groups(q, K, V, scale):
    q = np.asarray(q, dtype=np.float64)
    Hkv = K.shape[1]
    return np.stack([_orig_attention_one(q[h], K[:, h % Hkv], V[:, h % Hkv], scale) for h in range(q.shape[0])])


_orig_attention_one = A.attention_one
_orig_decode_attention = A.decode_attention

MUTANTS = {
    "scale dropped": [(A, "attention_one", _attention_no_scale)],
    "softmax not normalised": [(A, "attention_one", _attention_unnormalised)],
    "keys and values swapped": [(A, "decode_attention", _decode_attention_kv_swapped)],
    "query groups interleaved": [(A, "decode_attention", _decode_attention_modulo_groups)],
    "window keeps W+1 rows": [(Dm, "window_lo", lambda L, W: 0 if not W or W <= 0 else max(0, L - W - 1))],
    "window keeps W-1 rows": [(Dm, "window_lo", lambda L, W: 0 if not W or W <= 0 else max(0, L - W + 1))],
    "gather starts one row late": [(Dm, "gather_block", lambda row, P, lo, hi: A.gather_block(row, P, min(lo + 1, hi - 1), hi))],
    "one sink row too many": [(Dm, "_span", lambda L, W, S: _orig_span(L, W, S + 1 if S else 0))],
    "window part keeps W rows after the sinks": [(Dm, "_span", lambda L, W, S: (
        min(S, A.window_lo(L, W)), A.window_lo(L, W), max(0, L + 1 - W)) if W and W > 0 else (0, 0, 0))],
    "sink rows not attended": [(Dm, "_span", lambda L, W, S: (0,) + _orig_span(L, W, S)[1:])],
}

_orig_span = Dm._span


@pytest.mark.parametrize("name", list(MUTANTS))
def test_attention_mutant_is_caught(name, monkeypatch):
    for mod, attr, fn in MUTANTS[name]:
        monkeypatch.setattr(mod, attr, fn)
    try:
        problems = all_attention_problems()
    except Exception as e:
        problems = [repr(e)]
    assert problems, f"mutant '{name}' survived every pin"


def test_decode_loop_mutants_are_caught():
    # Pages outside the window never released, and the trim point one token late.
    class NoTrim(PageTable):
        def trim(self, rid, keep_from):
            return []

    class TrimLate(PageTable):
        def trim(self, rid, keep_from):
            return super().trim(rid, keep_from + 1)

    for cls in (NoTrim, TrimLate):
        try:
            problems = check_decode_page_counts(cls)
        except IndexError as e:  # reading a released page is a catch too
            problems = [repr(e)]
        assert problems, f"{cls.__name__} survived"


def test_sink_trim_mutants_are_caught():
    # The sink pages released with the rest, and the sink pages never trimmed past.
    class SinksReleased(PageTable):
        def trim(self, rid, keep_from, sink_rows=0):
            return super().trim(rid, keep_from)

    class NoTrimWithSinks(PageTable):
        def trim(self, rid, keep_from, sink_rows=0):
            return super().trim(rid, keep_from, sink_rows) if not sink_rows else []

    for cls in (SinksReleased, NoTrimWithSinks):
        try:
            problems = check_sink_page_counts(cls)
        except IndexError as e:
            problems = [repr(e)]
        assert problems, f"{cls.__name__} survived"
