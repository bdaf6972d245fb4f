"""Drive the product path and the oracle side by side on one workload.

``ProductSession`` uses only the library (host bookkeeping in C++, device
writes and attention through the C ABI); ``OracleSession`` uses only
``oracle/``. Both take the same seeded inputs from the workload generator:
the product generates its K/V/Q rows on the GPU, the oracle on the CPU (the
generator is bit-identical on both devices).
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle.attention as OA
from oracle.pagetable import PageTable
from oracle.raw_locations import RawLocationTable, align32
from paged_decode_attention_store_gb300 import workloads as wl

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


class ProductSession:
    def __init__(self, kb, w, device, max_requests, cols=None, mode="block", layers=None, seed=0):
        self.kb, self.w, self.dev, self.mode, self.seed = kb, w, device, mode, seed
        self.P = w.P
        self.layers = layers or w.layers
        self.dt = TORCH_DT[w.dtype]
        kdt = kb.KVP_BF16 if w.dtype == "bf16" else kb.KVP_F32
        extra = 1 if mode == "raw" else 0  # the dummy page of the raw-location layout
        self.kv = torch.zeros((2, self.layers, w.num_pages + extra, w.P, w.Hkv, w.D), dtype=self.dt, device=device)
        self.pool = kb.Pool(self.kv, w.P, kdt)
        self.host = kb.HostPageTable(w.num_pages, w.P, max_requests, w.free_order)
        self.max_requests = max_requests
        if mode == "block":
            cols = cols or 1
            self.table = torch.full((max_requests, cols), -1, dtype=torch.int32, device=device)
        else:
            cols = align32(min(cols or w.num_pages * w.P, w.num_pages * w.P))
            self.table = torch.zeros((max_requests + 1, cols), dtype=torch.int32, device=device)
            self.table[max_requests].fill_(w.num_pages * w.P)
        self.ws = None
        self.n_copies = 0

    def _i32(self, xs):
        return torch.tensor(list(xs), dtype=torch.int32, device=self.dev)

    def _write(self, writes):
        if not writes:
            return
        r, c, v = zip(*writes)
        self.kb.page_table_write(self.table, self._i32(r), self._i32(c), self._i32(v),
                                 expand=self.P if self.mode == "raw" else 1, error_word=self.pool.error_word)

    def new(self, rid):
        self.host.new(rid)

    def fork(self, src, dst):
        self._write(self.host.fork(src, dst))

    def release(self, rid):
        self.host.release(rid)

    def append(self, rids, positions):
        """Append one token per entry; K/V of (rid, position) come from the generator."""
        slots, writes, cows = self.host.append(rids)
        self._write(writes)
        if cows:
            s, d = zip(*cows)
            self.kb.copy_pages(self.pool, self._i32(s), self._i32(d))
            self.n_copies += len(cows)
        out_loc = self._i32(slots)
        for layer in range(self.layers):
            k, v = wl.kv_rows(self.seed, layer, rids, positions, self.w.Hkv, self.w.D, dtype=self.dt, device=self.dev)
            self.kb.store_cache(self.pool, layer, k, v, out_loc)
        return slots

    def trim(self, rid, keep_from, sinks=0):
        self._write(self.host.trim(rid, keep_from, sinks=sinks))

    def attend(self, layer, rids, lens, window, step, scale=None, table_rows=True, sinks=0):
        B = len(rids)
        if self.ws is None or self.ws_batch < B:
            self.ws = self.kb.alloc_workspace(self.pool, B, self.w.Hq, device=self.dev)
            self.ws_batch = B
        q = wl.q_rows(self.seed, step, layer, rids, self.w.Hq, self.w.D, dtype=self.dt, device=self.dev)
        out = torch.empty_like(q)
        scale = self.w.scale if scale is None else scale
        self.kb.paged_decode_attention(
            self.pool, layer, q, self.table,
            self.kb.KVP_RAW_LOCATIONS if self.mode == "raw" else self.kb.KVP_BLOCK_TABLE,
            self._i32(lens), window, scale, out, self.ws,
            table_rows=self._i32(rids) if table_rows else None, sinks=sinks)
        return out

    def gather(self, rids, lens, window, max_tokens, sinks=0):
        out = torch.empty((len(rids), max_tokens), dtype=torch.int32, device=self.dev)
        self.kb.gather_indices(self.pool, self.table,
                               self.kb.KVP_RAW_LOCATIONS if self.mode == "raw" else self.kb.KVP_BLOCK_TABLE,
                               self._i32(lens), window, out, table_rows=self._i32(rids), sinks=sinks)
        return out

    def error(self):
        return self.kb.kvp_sync_error(self.pool)


class OracleSession:
    """``raw_from_pages``: in raw mode, take a request's raw row as its block
    row expanded to tokens (``PageTable.raw_row``) instead of running the
    mini-sglang allocator, which has no window trim: needed once trims hand
    pages back to the free list."""

    def __init__(self, w, max_requests, mode="block", layers=None, seed=0, track=None, raw_cols=None,
                 raw_from_pages=False):
        self.w, self.mode, self.seed = w, mode, seed
        self.P = w.P
        self.layers = layers or w.layers
        self.pt = PageTable(w.num_pages, w.P, free_order=w.free_order)
        self.raw = None
        self.raw_from_pages = raw_from_pages
        if mode == "raw" and not raw_from_pages:
            self.raw = RawLocationTable(w.num_pages, w.P, max_requests, raw_cols or w.num_pages * w.P,
                                        free_page_order=w.free_order)
        self.stores = [OA.SlotStore() for _ in range(self.layers)]
        self.track = track  # rids whose rows are stored (None: all)
        self.dt = TORCH_DT[w.dtype]

    def new(self, rid):
        self.pt.new(rid)

    def fork(self, src, dst):
        self.pt.fork(src, dst)

    def release(self, rid):
        self.pt.release(rid)

    def append(self, rids, positions):
        before = {r: self.pt.length[r] for r in set(rids)}
        res = [self.pt.append(r) for r in rids]
        if self.raw is not None:
            # one allocation call for the whole batch, requests in first-seen order
            order, seen = [], set()
            for r in rids:
                if r not in seen:
                    seen.add(r)
                    order.append(r)
            self.raw.allocate_paged([(r, before[r], self.pt.length[r]) for r in order])
        for r in res:
            if r["cow"] is not None:
                for st in self.stores:
                    st.copy_page(r["cow"][0], r["cow"][1], self.P)
        keep = [i for i, r in enumerate(rids) if self.track is None or r in self.track]
        if keep:
            kr = [rids[i] for i in keep]
            kp = [positions[i] for i in keep]
            slots = [res[i]["slot"] for i in keep]
            for layer, st in enumerate(self.stores):
                k, v = wl.kv_rows(self.seed, layer, kr, kp, self.w.Hkv, self.w.D, dtype=self.dt)
                st.store_cache(slots, k.float().numpy(), v.float().numpy())
        return [r["slot"] for r in res]

    def trim(self, rid, keep_from, sinks=0):
        if sinks:
            return self.pt.trim(rid, keep_from, sink_rows=sinks)
        return self.pt.trim(rid, keep_from)

    def slots(self, rid, lo, L):
        if self.mode == "raw" and self.raw_from_pages:
            return OA.gather_raw(self.pt.raw_row(rid), lo, L)
        if self.mode == "raw":
            return OA.gather_raw(self.raw.page_table[rid], lo, L)
        return OA.gather_block(self.pt.block_row(rid), self.P, lo, L)

    def span_slots(self, rid, L, window, sinks):
        """Slots of every position the step attends (sink rows first)."""
        sink_end, lo = OA.sink_window(L, window, sinks)
        return self.slots(rid, 0, sink_end) + self.slots(rid, lo, L)

    def attend(self, layer, rid, L, window, step, scale=None, sinks=0):
        q = wl.q_rows(self.seed, step, layer, [rid], self.w.Hq, self.w.D, dtype=self.dt)[0].float().numpy()
        scale = self.w.scale if scale is None else scale
        if sinks:
            return OA.attend_request(self.stores[layer], q, self.span_slots(rid, L, window, sinks), scale)
        lo = OA.window_lo(L, window)
        return OA.attend_request(self.stores[layer], q, self.slots(rid, lo, L), scale)

    def table_row(self, rid):
        """The device-visible prefix of this request's table row."""
        if self.mode == "raw" and self.raw_from_pages:
            return self.pt.raw_row(rid)
        if self.mode == "raw":
            n = len(self.pt.block_row(rid)) * self.P
            return [int(x) for x in self.raw.page_table[rid, :n]]
        return self.pt.block_row(rid)


def tol_for(dtype):
    return 2e-2 if dtype == "bf16" else 1e-5


# bf16 outputs are also held to a bound relative to the request's largest
# output: max |gpu - oracle| <= REL_K * 2^-8 * max |oracle|. The GPU rounds
# the softmax weights and the output to bf16 (2^-9 relative each); the
# absolute 2e-2 alone lets a long context lose a 16-row page unseen, since
# outputs shrink like 1/sqrt(L). The largest ratio each test saw is printed
# at the end of the run.
REL_K = 2.0
RATIOS = {}


def close(got, ref, dtype, what=""):
    """Assert a GPU output against the oracle's: the absolute bound of its
    dtype and, for bf16, the relative bound above."""
    import os

    d = max_abs(got, ref)
    assert d <= tol_for(dtype), f"{what}: max |gpu - oracle| {d}"
    if dtype == "bf16":
        m = float(np.max(np.abs(np.asarray(ref, dtype=np.float64))))
        ratio = d / (2.0 ** -8 * m) if m > 0 else (0.0 if d == 0 else float("inf"))
        key = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        RATIOS[key] = max(RATIOS.get(key, 0.0), ratio)
        assert ratio <= REL_K, f"{what}: max |gpu - oracle| {d} = {ratio:.3f} x 2^-8 max|oracle| ({m})"


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def scale_of(D):
    return 1.0 / math.sqrt(D)
