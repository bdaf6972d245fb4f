"""PagedKVCache: the per-step driver a caller uses (one GPU, one process).

It owns a KV buffer in the mini-sglang layout (2, layers, pages, page_size,
kv_heads, head_dim), the C++ host bookkeeping and the device table, and
issues one decode step as the pages describe it:

1. host bookkeeping appends one token per request (a fresh page on a page
   boundary, lazy copy-on-write of a shared tail page, chapter 15 of
   silicon_compiler_from_scratch, section "The model");
2. the new table entries go to the device in one scatter (mini-sglang code
   series, part 4, with the page->token expansion done on the device for a
   raw-location table), copied-on-write pages are copied;
3. store_cache writes the new K/V rows of every layer to their slots;
4. paged_decode_attention reads each request's window through the table.

Host->device traffic per step is the table writes and slots (from pinned
staging buffers); everything else stays on the device.
"""

from __future__ import annotations

import torch

from . import binding as kb

_DT = {"bf16": (torch.bfloat16, kb.KVP_BF16), "f32": (torch.float32, kb.KVP_F32)}


def _align32(n):
    return (n + 31) // 32 * 32


class PagedKVCache:
    def __init__(self, num_pages, page_size, kv_heads, head_dim, num_layers, dtype="bf16", max_requests=256,
                 table_mode="block", max_seq_len=None, free_stack=None, device="cuda", zero=True):
        self.P, self.Hkv, self.D, self.layers = page_size, kv_heads, head_dim, num_layers
        self.num_pages = num_pages
        self.tdt, kdt = _DT[dtype]
        self.mode = table_mode
        self.raw = table_mode == "raw"
        self.dev = torch.device(device)
        extra = 1 if self.raw else 0  # dummy page of the raw-location layout
        alloc = torch.zeros if zero else torch.empty
        self.kv = alloc((2, num_layers, num_pages + extra, page_size, kv_heads, head_dim), dtype=self.tdt,
                        device=self.dev)
        self.pool = kb.Pool(self.kv, page_size, kdt)
        self.host = kb.HostPageTable(num_pages, page_size, max_requests, free_stack)
        self.max_requests = max_requests
        max_seq_len = max_seq_len or num_pages * page_size
        if self.raw:
            cols = _align32(min(max_seq_len, num_pages * page_size))
            self.table = torch.zeros((max_requests + 1, cols), dtype=torch.int32, device=self.dev)
            self.table[max_requests].fill_(num_pages * page_size)  # dummy row -> dummy page
        else:
            cols = -(-max_seq_len // page_size)
            self.table = torch.full((max_requests, cols), -1, dtype=torch.int32, device=self.dev)
        self.table_mode = kb.KVP_RAW_LOCATIONS if self.raw else kb.KVP_BLOCK_TABLE
        self._ws = {}
        self.copies = 0
        self.h2d_bytes = 0  # bytes this driver has copied host -> device

    # -- host-side staging -------------------------------------------------
    def _to_device(self, flat):
        # A fresh pinned block per call: torch's caching host allocator does
        # not hand it out again before the asynchronous copy has completed.
        host = torch.tensor(flat, dtype=torch.int32).pin_memory()
        self.h2d_bytes += 4 * len(flat)
        return host.to(self.dev, non_blocking=True)

    def _write_table(self, writes):
        if not writes:
            return
        r, c, v = zip(*writes)
        d = self._to_device(list(r) + list(c) + list(v))
        n = len(writes)
        kb.page_table_write(self.table, d[:n], d[n:2 * n], d[2 * n:], expand=self.P if self.raw else 1,
                            error_word=self.pool.error_word)

    # -- request lifecycle ---------------------------------------------------
    def new(self, rid):
        self.host.new(rid)

    def fork(self, src, dst):
        self._write_table(self.host.fork(src, dst))

    def release(self, rid):
        self.host.release(rid)

    def trim(self, rid, keep_from):
        """Release front pages below keep_from; returns the number of table writes."""
        writes = self.host.trim(rid, keep_from)
        self._write_table(writes)
        return len(writes)

    def append(self, rids):
        """Host bookkeeping for one token per entry; returns the slots on the device.

        Also leaves the counts of this call's table writes and copies in
        ``last_writes`` / ``last_copies``."""
        slots, writes, cows = self.host.append(rids)
        self.last_writes, self.last_copies = len(writes), len(cows)
        n, nw, nc = len(slots), len(writes), len(cows)
        flat = list(slots)
        if nw:
            r, c, v = zip(*writes)
            flat += list(r) + list(c) + list(v)
        if nc:
            s, d = zip(*cows)
            flat += list(s) + list(d)
        dev = self._to_device(flat)
        if nw:
            kb.page_table_write(self.table, dev[n:n + nw], dev[n + nw:n + 2 * nw], dev[n + 2 * nw:n + 3 * nw],
                                expand=self.P if self.raw else 1, error_word=self.pool.error_word)
        if nc:
            o = n + 3 * nw
            kb.copy_pages(self.pool, dev[o:o + nc], dev[o + nc:o + 2 * nc])
            self.copies += nc
        return dev[:n]

    def store(self, layer, k, v, out_loc):
        kb.store_cache(self.pool, layer, k, v, out_loc)

    def workspace(self, batch, num_q_heads):
        key = (batch, num_q_heads)
        if key not in self._ws:
            self._ws[key] = kb.alloc_workspace(self.pool, batch, num_q_heads, device=self.dev)
        return self._ws[key]

    def attend(self, layer, q, context_lens, window, scale, out, table_rows=None):
        ws = self.workspace(q.shape[0], q.shape[1])
        kb.paged_decode_attention(self.pool, layer, q, self.table, self.table_mode, context_lens, window, scale,
                                  out, ws, table_rows=table_rows)

    def check(self):
        """Raise if a device-side error was recorded since the last check."""
        e = kb.kvp_sync_error(self.pool)
        if e != 0:
            raise kb.KvpError(e, "device")
