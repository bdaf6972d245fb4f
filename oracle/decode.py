"""One layer's decode loop over the oracle's tables (test infrastructure only).

Order of one step, for every request of the batch (reading of "A Paged KV
Cache and Sliding-Window Attention", chapter 15, section "The model", with
the attention moved after a separate store):

1. append the new token to the request's block table (a fresh page on a page
   boundary, lazy copy-on-write of a shared tail page) -> its slot;
2. copy every copied-on-write page, then store the new K/V rows at their
   slots (mini-sglang code series, part 4: ``store_cache`` with ``out_loc``);
3. attend positions ``max(0, L - W) .. L - 1`` (``L`` = length after the
   append) read through the table;
4. trim the request to ``keep_from = L + 1 - W`` so that the page holding the
   first row the NEXT step needs is kept.

With ``S`` attention sinks (chapter 15, exercise "Attention sinks") step 3
attends ``0 .. min(S, lo) - 1`` and ``lo .. L - 1`` with ``lo = max(0, L -
(W - S))``, and step 4 trims to ``keep_from = L + 1 - (W - S)`` keeping the
sink pages.
"""

from __future__ import annotations

import numpy as np

from .attention import SlotStore, attend_request, gather_block, window_lo


def _span(L: int, window, sinks: int):
    """(sink_end, lo, keep_from) of a step with context ``L``."""
    if window is None or window <= 0:
        return 0, 0, 0
    if sinks < 0 or sinks >= window:
        raise ValueError("sink rows must satisfy 0 <= S < W")
    lo = window_lo(L, window - sinks)
    return min(sinks, lo), lo, max(0, L + 1 - (window - sinks))


class BlockDecoder:
    """Decode loop in block-table mode (one layer)."""

    def __init__(self, pt, window, scale: float, sinks: int = 0):
        self.pt = pt
        self.P = pt.page
        self.window = window
        self.sinks = sinks
        self.scale = scale
        self.store = SlotStore()

    def _trim(self, rid) -> None:
        kf = _span(self.pt.length[rid], self.window, self.sinks)[2]
        if self.sinks:
            self.pt.trim(rid, kf, sink_rows=self.sinks)
        else:
            self.pt.trim(rid, kf)

    def prefill(self, rid, k, v) -> list:
        """Append ``len(k)`` rows to request ``rid`` (no attention); returns slots."""
        slots = []
        for i in range(len(k)):
            r = self.pt.append(rid)
            if r["cow"] is not None:
                self.store.copy_page(r["cow"][0], r["cow"][1], self.P)
            slots.append(r["slot"])
            self.store.store_cache([r["slot"]], k[i:i + 1], v[i:i + 1])
            if self.window is not None and self.window > 0:
                self._trim(rid)
        return slots

    def step(self, rids, q, k_new, v_new):
        """One decode step. Returns (slots, copy-on-write pairs, outputs [B, Hq, D])."""
        slots, cows = [], []
        for rid in rids:
            r = self.pt.append(rid)
            if r["cow"] is not None:
                cows.append(r["cow"])
            slots.append(r["slot"])
        for src, dst in cows:
            self.store.copy_page(src, dst, self.P)
        self.store.store_cache(slots, k_new, v_new)
        outs = []
        for i, rid in enumerate(rids):
            L = self.pt.length[rid]
            row = self.pt.block_row(rid)
            if self.sinks:
                sink_end, lo, _ = _span(L, self.window, self.sinks)
                s = gather_block(row, self.P, 0, sink_end) + gather_block(row, self.P, lo, L)
            else:
                s = gather_block(row, self.P, window_lo(L, self.window), L)
            outs.append(attend_request(self.store, q[i], s, self.scale))
        if self.window is not None and self.window > 0:
            for rid in rids:
                self._trim(rid)
        return slots, cows, np.stack(outs)

