"""Dense softmax decode-attention oracle (test infrastructure only; see ``oracle``).

"Week 3 Day 3: Paged KV Cache" (tiny-llm), section "Correctness Checkpoint:
Gather Pages for Dense Attention", keeps the pages as the source of truth,
gathers a request's rows back into dense K/V in logical order and feeds them
to the plain dense attention equation. The pages never print that equation,
so this module takes the textbook scaled-dot-product form, computed in
float64 on rows that are widened exactly from their stored type:

    s_t = scale * <q_h, k_t>          for the gathered positions t
    p   = softmax(s)                  (shifted by max(s) before exp)
    out = sum_t p_t * v_t

Which positions: "A Paged KV Cache and Sliding-Window Attention" (chapter
15, section "The model") lets a step with context ``L`` and window ``W``
attend the new token and at most ``W - 1`` earlier ones, i.e. positions
``L - min(L, W) … L - 1``. With the new token stored before the attention
runs, that is ``lo = max(0, L - W)`` up to ``L``; no window (``W`` absent or
``<= 0``) means ``lo = 0``.

Attention sinks: chapter 15's exercise "Attention sinks" keeps the first
``S`` rows as well and takes the last ``W - S`` for the rest, so the context
is still ``W`` rows: positions ``0 … min(S, lo) - 1`` and ``lo … L - 1`` with
``lo = max(0, L - (W - S))``. ``S = 0`` is the plain window; ``S`` must stay
below ``W`` (the new token is always attended).

Grouped-query heads: query head ``h`` reads KV head ``h // (Hq // Hkv)``
(contiguous groups); the pages do not state a mapping, this is the plain one.

Rows are read LITERALLY through the tables: a block table maps position
``t`` to slot ``table[t // P] * P + t % P`` ("PagedAttention block
allocator", section "Sequence block table"); a raw-location table maps it to
``table[t]`` (mini-sglang code series, part 4). A negative entry is a
released page and reading it is an error, never a mask.
"""

from __future__ import annotations

import numpy as np


def window_lo(L: int, W) -> int:
    """First position a step with context ``L`` attends under window ``W``."""
    if W is None or W <= 0:
        return 0
    return max(0, L - W)


def sink_window(L: int, W, S: int = 0):
    """(sink_end, lo): a step with context ``L``, window ``W`` and ``S`` sink
    rows attends ``0 <= t < sink_end`` and ``lo <= t < L``."""
    if W is None or W <= 0:
        return 0, 0
    if S < 0 or S >= W:
        raise ValueError("sink rows must satisfy 0 <= S < W")
    lo = window_lo(L, W - S)
    return min(S, lo), lo


def attended_positions(L: int, W, S: int = 0) -> list:
    """Every position a step with context ``L`` attends, in logical order."""
    sink_end, lo = sink_window(L, W, S)
    return list(range(0, sink_end)) + list(range(lo, L))


def verify_positions(L: int, M: int, W, S: int = 0) -> list:
    """Multi-token verify: the M newest tokens of a request with context L
    (positions L - M .. L - 1) are queries at once. Query j attends what a
    single-token step with context L - M + j + 1 attends (causal: nothing
    after its own position). Returns one position list per query."""
    if M < 1 or M > L:
        raise ValueError("need 1 <= M <= L")
    return [attended_positions(L - M + j + 1, W, S) for j in range(M)]


def attention_one(q, K, V, scale: float):
    """One query row against ``n >= 1`` key/value rows, float64.

    q: [D]; K, V: [n, D]. Returns [D].
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        raise ValueError("attention over zero rows")
    s = scale * (K @ q)
    s = s - s.max()
    w = np.exp(s)
    return (w @ V) / w.sum()


def decode_attention(q, K, V, scale: float):
    """All query heads of one request.

    q: [Hq, D]; K, V: [n, Hkv, D] in logical order. Returns [Hq, D] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    Hq = q.shape[0]
    Hkv = K.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    out = np.empty_like(q)
    for h in range(Hq):
        g = h // G
        out[h] = attention_one(q[h], K[:, g, :], V[:, g, :], scale)
    return out


def gather_block(table_row, P: int, lo: int, hi: int) -> list:
    """Slots of positions ``lo <= t < hi`` through a block-table row."""
    slots = []
    for t in range(lo, hi):
        page = int(table_row[t // P])
        if page < 0:
            raise IndexError(f"position {t} lies in a released page")
        slots.append(page * P + t % P)
    return slots


def gather_raw(raw_row, lo: int, hi: int) -> list:
    """Slots of positions ``lo <= t < hi`` through a raw-location row."""
    slots = []
    for t in range(lo, hi):
        s = int(raw_row[t])
        if s < 0:
            raise IndexError(f"position {t} lies in a released page")
        slots.append(s)
    return slots


class SlotStore:
    """One layer of the KV pool viewed as flat token slots (``page * P + offset``).

    Only slots that were written exist; reading any other slot is an error.
    ``store_cache`` follows the mini-sglang code series, part 4, section "KV
    버퍼는 6축인데, 쓸 때는 3축이다": row ``i`` of ``k`` and ``v`` goes to slot
    ``out_loc[i]``.
    """

    def __init__(self):
        self.k = {}
        self.v = {}

    def store_cache(self, out_loc, k, v) -> None:
        for i, s in enumerate(out_loc):
            self.k[int(s)] = np.array(k[i], dtype=np.float64)
            self.v[int(s)] = np.array(v[i], dtype=np.float64)

    def copy_page(self, src: int, dst: int, P: int) -> None:
        """Copy-on-write: the whole page ``src`` into page ``dst``."""
        for j in range(P):
            s, d = src * P + j, dst * P + j
            if s in self.k:
                self.k[d] = self.k[s].copy()
                self.v[d] = self.v[s].copy()
            else:
                self.k.pop(d, None)
                self.v.pop(d, None)

    def gather(self, slots):
        K = np.stack([self.k[s] for s in slots])
        V = np.stack([self.v[s] for s in slots])
        return K, V


def attend_request(store: SlotStore, q, slots, scale: float):
    """Decode attention of one request over the given slots (logical order)."""
    K, V = store.gather(slots)
    return decode_attention(q, K, V, scale)
