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

import ctypes

import numpy as np
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
        self._steps = {}
        self.lengths = np.zeros(max_requests, np.int64)  # tokens appended, per request (the caller's count)
        self.copies = 0
        self.h2d_bytes = 0  # bytes this driver has copied host -> device

    # -- host-side staging -------------------------------------------------
    def _to_device(self, flat):
        # A fresh pinned block per call: torch's caching host allocator does
        # not hand it out again before the asynchronous copy has completed.
        host = torch.from_numpy(np.ascontiguousarray(flat, dtype=np.int32)).pin_memory()
        self.h2d_bytes += 4 * host.numel()
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
        self.lengths[rid] = 0

    def fork(self, src, dst):
        self._write_table(self.host.fork(src, dst))
        self.lengths[dst] = self.lengths[src]

    def release(self, rid):
        self.host.release(rid)
        self.lengths[rid] = 0

    def trim(self, rid, keep_from, sinks=0):
        """Release the pages below keep_from (except the first ceil(sinks / P));
        returns the number of table writes."""
        writes = self.host.trim(rid, keep_from, sinks=sinks)
        self._write_table(writes)
        return len(writes)

    def append(self, rids):
        """Host bookkeeping for one token per entry; returns the slots on the device.

        Also leaves the counts of this call's table writes and copies in
        ``last_writes`` / ``last_copies``."""
        r = np.ascontiguousarray(rids, dtype=np.int32)
        n = int(r.shape[0])
        buf = np.empty(6 * max(n, 1), np.int32)  # slots, table writes (rows, cols, values), copy pairs
        slots, tw, cow = buf[:n], buf[n:4 * n].reshape(3, n), buf[4 * n:6 * n].reshape(2, n)
        nw, nc = self.host.append_into(r, slots, tw, cow)
        self.lengths += np.bincount(r, minlength=self.lengths.shape[0])
        self.last_writes, self.last_copies = nw, nc
        dev = self._to_device(np.concatenate((slots, tw[:, :nw].ravel(), cow[:, :nc].ravel())))
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

    def attend(self, layer, q, context_lens, window, scale, out, table_rows=None, sinks=0):
        ws = self.workspace(q.shape[0], q.shape[1])
        kb.paged_decode_attention(self.pool, layer, q, self.table, self.table_mode, context_lens, window, scale,
                                  out, ws, table_rows=table_rows, sinks=sinks)

    def store_and_attend(self, layer, q, k, v, out_loc, context_lens, window, scale, out, table_writes=None,
                         table_rows=None, sinks=0):
        """store_cache + paged_decode_attention of one layer in one launch;
        ``out_loc[b]`` must be the slot of request b's newest position, and
        ``table_writes`` (rows, cols, vals device tensors) may only add the
        pages of this step's new tokens."""
        ws = self.workspace(q.shape[0], q.shape[1])
        kb.store_cache_and_attention(self.pool, layer, q, k, v, out_loc, self.table, self.table_mode, context_lens,
                                     window, scale, out, ws, table_rows=table_rows, table_writes=table_writes,
                                     sinks=sinks)

    def verify(self, layer, q, context_lens, window, scale, out, table_rows=None, sinks=0):
        """Multi-token verify: q/out [B, M, Hq, D], query j of request b at
        position context_lens[b] - M + j (the M newest tokens, stored)."""
        B, M, Hq = q.shape[0], q.shape[1], q.shape[2]
        key = ("verify", B, M, Hq)
        if key not in self._ws:
            self._ws[key] = kb.alloc_verify_workspace(self.pool, B, M, Hq, device=self.dev)
        kb.paged_verify_attention(self.pool, layer, q, self.table, self.table_mode, context_lens, window, scale,
                                  out, self._ws[key], table_rows=table_rows, sinks=sinks)

    def rewind(self, rid, n):
        """Drop the newest n tokens of a request (rejected drafts); returns
        the number of pages given back."""
        writes = self.host.rewind(rid, n)
        self._write_table(writes)
        self.lengths[rid] -= n
        return len(writes)

    def prefill(self, layer, q, context_lens, window, scale, out, q_lens=None, table_rows=None, sinks=0):
        """Chunked prefill: q/out [B, C, Hq, D], query j of request b at
        position context_lens[b] - q_lens[b] + j (the chunk's rows stored)."""
        kb.paged_prefill_attention(self.pool, layer, q, self.table, self.table_mode, context_lens, window, scale,
                                   out, q_lens=q_lens, table_rows=table_rows, sinks=sinks)

    def prefill_step(self, rids, q, k, v, out, window, scale, sinks=0):
        """One chunked-prefill step for ``rids``, all layers: append each
        request's C new tokens (host bookkeeping, table writes, copy-on-write),
        store their K/V and attend them at once. ``q``/``out`` [layers][B, C,
        Hq, D], ``k``/``v`` [layers][B * C, Hkv, D] (request-major), on the host
        (pinned) or the device; returns when ``out`` holds the results."""
        self._multi_step("prefill", rids, q, k, v, out, window, scale, sinks)

    def verify_step(self, rids, q, k, v, out, window, scale, sinks=0):
        """One speculative-decoding verify step for requests ``rids`` (ids =
        table rows), all layers: append the M drafted tokens of each request
        (host bookkeeping, table writes, copy-on-write), store their K/V rows
        and verify them. ``q``/``out`` [layers][B, M, Hq, D] and ``k``/``v``
        [layers][B * M, Hkv, D] (request-major) on the host (pinned) or the
        device. Returns when ``out`` holds the results; the caller then
        rewinds the rejected drafts with :meth:`rewind`."""
        self._multi_step("verify", rids, q, k, v, out, window, scale, sinks)

    def _multi_step(self, kind, rids, q, k, v, out, window, scale, sinks):
        B, M = q[0].shape[0], q[0].shape[1]
        main = torch.cuda.current_stream(self.dev)
        staged = None
        if not q[0].is_cuda:
            # host inputs: every layer's q/k/v go up on a side stream right away,
            # while the host bookkeeping below runs; layer l's store waits for
            # layer l's copies only
            side = self._steps.get("multi_h2d")
            if side is None:
                side = self._steps["multi_h2d"] = torch.cuda.Stream(self.dev)
            side.wait_stream(main)
            staged = []
            with torch.cuda.stream(side):
                for layer in range(self.layers):
                    xs = tuple(x[layer].to(self.dev, non_blocking=True) for x in (q, k, v))
                    for t in xs:
                        t.record_stream(main)
                    ev = torch.cuda.Event()
                    ev.record(side)
                    staged.append((xs, ev))
                    self.h2d_bytes += sum(x[layer].numel() * x[layer].element_size() for x in (q, k, v))
        r = np.ascontiguousarray(rids, dtype=np.int32)
        ctx = self.lengths[r] + M
        out_loc = self.append(np.repeat(r, M))
        lens = self._to_device(ctx)
        rows = self._to_device(r)
        host_out = not out[0].is_cuda
        for layer in range(self.layers):
            if staged is None:
                qd, kd, vd = (x[layer] for x in (q, k, v))
            else:
                (qd, kd, vd), ev = staged[layer]
                main.wait_event(ev)
            self.store(layer, kd, vd, out_loc)
            od = torch.empty_like(qd) if host_out else out[layer]
            if kind == "verify":
                self.verify(layer, qd, lens, window, scale, od, table_rows=rows, sinks=sinks)
            else:
                self.prefill(layer, qd, lens, window, scale, od, table_rows=rows, sinks=sinks)
            if host_out:
                out[layer].copy_(od, non_blocking=True)
        torch.cuda.current_stream(self.dev).synchronize()

    def check(self):
        """Raise if a device-side error was recorded since the last check."""
        e = kb.kvp_sync_error(self.pool)
        if e != 0:
            raise kb.KvpError(e, "device")


    # -- one decode step, host buffers in and out ----------------------------
    def decode_step(self, rids, q, k, v, out, window, scale, sinks=0):
        """One decode step for the requests ``rids`` (one token each; request
        id = table row), through the native kvp_decode_step.

        ``q`` [layers][B, Hq, D], ``k``/``v`` [layers][B, Hkv, D] and ``out``
        [layers][B, Hq, D] are lists of tensors, all on the host (pinned) or
        all on the device. With several layers, host inputs are copied per
        layer on a side stream and each layer's store + attention waits only
        for its own inputs, and each output is copied back on another side
        stream as soon as its layer is done; a single layer copies on the
        step's own stream. Returns when ``out`` holds the results.
        """
        L = kb.lib()
        n = len(rids)
        Hq = q[0].shape[1]
        st = self._step_state(n, Hq)
        rids = np.ascontiguousarray(rids, dtype=np.int32)
        stream = torch.cuda.current_stream(self.dev)
        slot = st["ring"][st["next"]]
        st["next"] ^= 1
        slot["event"].synchronize()  # its previous copy has finished reading it
        host_io = not q[0].is_cuda
        vp = ctypes.c_void_p
        arr = lambda ts: (vp * self.layers)(*[t.data_ptr() for t in ts])  # noqa: E731
        ready = done = None
        if host_io:
            qd, kd, vd = st["in"]
            od = st["out"]
            qp, kp, vpp, op = st["in_p"][0], st["in_p"][1], st["in_p"][2], st["out_p"]
            side = self.layers > 1  # overlap the per-layer copies with the other layers' kernels
            cs = st["h2d"] if side else stream
            if side:
                st["h2d"].wait_stream(stream)  # the previous step's kernels are done with the buffers
            with torch.cuda.stream(cs):
                for layer in range(self.layers):
                    qd[layer].copy_(q[layer], non_blocking=True)
                    kd[layer].copy_(k[layer], non_blocking=True)
                    vd[layer].copy_(v[layer], non_blocking=True)
                    if side:
                        st["ready"][layer].record(cs)
            self.h2d_bytes += sum(t[i].numel() * t[i].element_size() for t in (q, k, v) for i in range(self.layers))
            if side:
                ready, done = st["ready_p"], st["done_p"]
        else:
            side = False
            qp, kp, vpp, op = arr(q), arr(k), arr(v), arr(out)
        info = kb.StepInfo()
        ws = self.workspace(n, Hq)
        kb._check(L.kvp_decode_step(self.host.handle, self.pool.handle, vp(self.table.data_ptr()), self.table.shape[0],
                                    self.table.shape[1], self.table_mode, rids.ctypes.data_as(vp), n,
                                    int(window or 0), int(sinks), Hq, float(scale), qp, kp, vpp, op, ready,
                                    done, vp(slot["host"].data_ptr()), vp(st["dev"].data_ptr()), st["cap"],
                                    vp(ws.data_ptr()), ws.numel(), vp(stream.cuda_stream), ctypes.byref(info)),
                  "kvp_decode_step")
        slot["event"].record(stream)
        self.h2d_bytes += 4 * info.meta_ints
        self.last_writes, self.last_copies, self.last_trims = info.n_table_writes, info.n_copies, info.n_trim_writes
        self.copies += info.n_copies
        np.add.at(self.lengths, rids, 1)
        if host_io:
            if side:
                with torch.cuda.stream(st["d2h"]):
                    for layer in range(self.layers):
                        st["d2h"].wait_event(st["done"][layer])
                        out[layer].copy_(od[layer], non_blocking=True)
                st["d2h"].synchronize()
            else:
                for layer in range(self.layers):
                    out[layer].copy_(od[layer], non_blocking=True)
        stream.synchronize()  # the step's outputs are in `out`
        return 4 * info.meta_ints

    def _step_state(self, n, Hq):
        key = (n, Hq)
        st = self._steps.get(key)
        if st is not None:
            return st
        cap = 8 * n + 3 * (4 * n + 64)
        ring = []
        for _ in range(2):
            host = torch.zeros(cap, dtype=torch.int32, pin_memory=True)
            ev = torch.cuda.Event()
            ev.record(torch.cuda.current_stream(self.dev))
            ring.append({"host": host, "event": ev})
        ready = [torch.cuda.Event() for _ in range(self.layers)]
        done = [torch.cuda.Event() for _ in range(self.layers)]
        for e in ready + done:  # torch creates the CUDA event at its first record
            e.record(torch.cuda.current_stream(self.dev))
        vp = ctypes.c_void_p
        st = {
            "cap": cap, "ring": ring, "next": 0,
            "dev": torch.empty(cap, dtype=torch.int32, device=self.dev),
            "in": [[torch.empty((n, Hq, self.D), dtype=self.tdt, device=self.dev) for _ in range(self.layers)],
                   [torch.empty((n, self.Hkv, self.D), dtype=self.tdt, device=self.dev) for _ in range(self.layers)],
                   [torch.empty((n, self.Hkv, self.D), dtype=self.tdt, device=self.dev) for _ in range(self.layers)]],
            "out": [torch.empty((n, Hq, self.D), dtype=self.tdt, device=self.dev) for _ in range(self.layers)],
            "h2d": torch.cuda.Stream(self.dev), "d2h": torch.cuda.Stream(self.dev),
            "ready": ready, "done": done,
            "ready_p": (vp * self.layers)(*[e.cuda_event for e in ready]),
            "done_p": (vp * self.layers)(*[e.cuda_event for e in done]),
        }
        st["in_p"] = [(vp * self.layers)(*[t.data_ptr() for t in ts]) for ts in st["in"]]
        st["out_p"] = (vp * self.layers)(*[t.data_ptr() for t in st["out"]])
        torch.cuda.synchronize(self.dev)
        self._steps[key] = st
        return st


class DevicePagedKVCache:
    """A paged KV cache whose page bookkeeping lives on the device (kvp_dev_*).

    The same layout as :class:`PagedKVCache` (mini-sglang's 6-axis buffer, a
    block table or a raw-location table); the free list, reference counts
    and lengths are device arrays, so a decode step (:meth:`decode_step`)
    makes no host decision and copies nothing to the device but q/k/v.
    Request ids are table rows. Lengths are not mirrored on the host: the
    caller knows its own schedule.
    """

    def __init__(self, num_pages, page_size, kv_heads, head_dim, num_layers, dtype="bf16", max_requests=256,
                 table_mode="block", max_seq_len=None, free_stack=None, device="cuda", zero=True):
        self.P, self.Hkv, self.D, self.layers = page_size, kv_heads, head_dim, num_layers
        self.num_pages = num_pages
        self.tdt, kdt = _DT[dtype]
        self.raw = table_mode == "raw"
        self.dev = torch.device(device)
        extra = 1 if self.raw else 0
        alloc = torch.zeros if zero else torch.empty
        self.kv = alloc((2, num_layers, num_pages + extra, page_size, kv_heads, head_dim), dtype=self.tdt,
                        device=self.dev)
        self.pool = kb.Pool(self.kv, page_size, kdt)
        max_seq_len = max_seq_len or num_pages * page_size
        if self.raw:
            cols = _align32(min(max_seq_len, num_pages * page_size))
            self.table = torch.zeros((max_requests + 1, cols), dtype=torch.int32, device=self.dev)
            self.table[max_requests].fill_(num_pages * page_size)  # dummy row -> dummy page
        else:
            cols = -(-max_seq_len // page_size)
            self.table = torch.full((max_requests, cols), -1, dtype=torch.int32, device=self.dev)
        self.table_mode = kb.KVP_RAW_LOCATIONS if self.raw else kb.KVP_BLOCK_TABLE
        self.pages = kb.DevicePages(num_pages, page_size, max_requests, self.table, self.table_mode,
                                    free_stack=free_stack, device=self.dev)
        self.may_share = False  # set by fork: appends may then copy shared tail pages
        self._ws = {}
        self._scratch = {}
        self._staging = {}
        self._ptrs = {}

    def _i32(self, xs):
        return torch.as_tensor(list(xs), dtype=torch.int32).to(self.dev, non_blocking=True)

    def new(self, rids):
        self.pages.new(self._i32(rids))

    def append(self, rids, counts=None):
        """Append counts[i] rows (default one) to each request; returns the
        slots of the new rows on the device (request-major), after copying
        any shared tail page."""
        n = len(rids)
        total = n if counts is None else int(sum(counts))
        out_loc = torch.empty(max(total, 1), dtype=torch.int32, device=self.dev)
        cow = torch.empty((2, n), dtype=torch.int32, device=self.dev)
        n_cow = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.pages.append(self._i32(rids), out_loc, cow[0], cow[1], n_cow,
                          counts=None if counts is None else self._i32(counts))
        if self.may_share:
            kb.copy_pages_device_count(self.pool, cow[0], cow[1], n_cow)
        return out_loc[:total]

    def store(self, layer, k, v, out_loc):
        kb.store_cache(self.pool, layer, k, v, out_loc)

    def fork(self, src, dst):
        self.pages.fork(self._i32(src), self._i32(dst))
        self.may_share = True

    def trim(self, rids, window, sinks=0):
        self.pages.trim(self._i32(rids), window=window, sinks=sinks)

    def release(self, rids):
        self.pages.release(self._i32(rids))

    def rewind(self, rids, n_back):
        """Drop the newest n_back[i] rows of each request (rejected drafts)."""
        self.pages.rewind(self._i32(rids), self._i32(n_back))

    def workspace(self, batch, num_q_heads, num_q_tokens=1):
        key = (batch, num_q_heads, num_q_tokens)
        if key not in self._ws:
            self._ws[key] = (kb.alloc_workspace(self.pool, batch, num_q_heads, device=self.dev) if num_q_tokens == 1
                             else kb.alloc_verify_workspace(self.pool, batch, num_q_tokens, num_q_heads,
                                                            device=self.dev))
        return self._ws[key]

    def verify(self, layer, q, context_lens, window, scale, out, table_rows=None, sinks=0):
        """Multi-token verify attention: q/out [B, M, Hq, D] (the M newest tokens, stored)."""
        ws = self.workspace(q.shape[0], q.shape[2], q.shape[1])
        kb.paged_verify_attention(self.pool, layer, q, self.table, self.table_mode, context_lens, window, scale,
                                  out, ws, table_rows=table_rows, sinks=sinks)

    def attend(self, layer, q, context_lens, window, scale, out, table_rows=None, sinks=0):
        ws = self.workspace(q.shape[0], q.shape[1])
        kb.paged_decode_attention(self.pool, layer, q, self.table, self.table_mode, context_lens, window, scale,
                                  out, ws, table_rows=table_rows, sinks=sinks)

    def decode_step(self, rids, q, k, v, out, window, scale, sinks=0):
        """One decode step, all layers, through kvp_decode_step_device.
        ``rids``: device int32 [B]; q/k/v/out: per-layer DEVICE tensors
        ([B, Hq, D] and [B, Hkv, D]). Asynchronous: nothing is synchronised."""
        n, Hq = rids.numel(), q[0].shape[1]
        scratch = self._scratch.get(n)
        if scratch is None:
            scratch = self._scratch[n] = torch.zeros(4 * n + 1, dtype=torch.int32, device=self.dev)
        ws = self.workspace(n, Hq)
        vp = ctypes.c_void_p
        arr = lambda ts: (vp * self.layers)(*[t.data_ptr() for t in ts])  # noqa: E731
        stream = torch.cuda.current_stream(self.dev)
        kb._check(kb.lib().kvp_decode_step_device(
            self.pages.handle, self.pool.handle, vp(self.table.data_ptr()), self.table.shape[0], self.table.shape[1],
            self.table_mode, vp(rids.data_ptr()), n, int(window or 0), int(sinks), Hq, float(scale), arr(q), arr(k),
            arr(v), arr(out), None, None, vp(scratch.data_ptr()), int(self.may_share), vp(ws.data_ptr()),
            ws.numel(), vp(stream.cuda_stream)), "kvp_decode_step_device")

    def _ptr_array(self, ts):
        """ctypes array of the tensors' data pointers, cached by their addresses."""
        key = tuple(t.data_ptr() for t in ts)
        arr = self._ptrs.get(key)
        if arr is None:
            if len(self._ptrs) > 256:
                self._ptrs.clear()
            arr = self._ptrs[key] = (ctypes.c_void_p * len(ts))(*key)
        return arr

    def decode_step_host(self, rids, q, k, v, out, window, scale, sinks=0):
        """One decode step with HOST buffers (pinned): ``q``/``k``/``v``/``out``
        are per-layer host tensors; inputs are copied to device staging, the
        step runs with the bookkeeping on the device, outputs come back. One
        native call (kvp_decode_step_device_io); returns when ``out`` holds
        the results. ``rids``: device int32 [B]."""
        n, Hq = rids.numel(), q[0].shape[1]
        key = (n, Hq)
        stage = self._staging.get(key)
        if stage is None:
            mk = lambda t: torch.empty(t.shape, dtype=t.dtype, device=self.dev)  # noqa: E731
            stage = self._staging[key] = ([mk(t) for t in q], [mk(t) for t in k], [mk(t) for t in v],
                                          [mk(t) for t in out], torch.zeros(4 * n + 1, dtype=torch.int32,
                                                                            device=self.dev))
        qd, kd, vd, od, scratch = stage
        ws = self.workspace(n, Hq)
        vp = ctypes.c_void_p
        pa = self._ptr_array
        stream = torch.cuda.current_stream(self.dev)
        kb._check(kb.lib().kvp_decode_step_device_io(
            self.pages.handle, self.pool.handle, vp(self.table.data_ptr()), self.table.shape[0], self.table.shape[1],
            self.table_mode, vp(rids.data_ptr()), n, int(window or 0), int(sinks), Hq, float(scale), pa(q), pa(k),
            pa(v), pa(out), pa(qd), pa(kd), pa(vd), pa(od), vp(scratch.data_ptr()), int(self.may_share),
            vp(ws.data_ptr()), ws.numel(), vp(stream.cuda_stream)), "kvp_decode_step_device_io")

    def verify_step_host(self, rids, q, k, v, n_back, out, window, scale, sinks=0):
        """One speculative-decoding verify step with HOST buffers (pinned),
        the page bookkeeping on the device: the M drafts of every request are
        appended, stored and verified at once, then each request's rejected
        drafts (``n_back``: host int32 [B], 0..M) are rewound. ``q``/``out``
        per-layer host tensors [B, M, Hq, D], ``k``/``v`` [B * M, Hkv, D]
        (request-major); ``rids``: device int32 [B]. One native call
        (kvp_verify_step_device_io); returns when ``out`` holds the results."""
        n, M, Hq = rids.numel(), q[0].shape[1], q[0].shape[2]
        key = ("verify", n, M, Hq)
        stage = self._staging.get(key)
        if stage is None:
            mk = lambda t: torch.empty(t.shape, dtype=t.dtype, device=self.dev)  # noqa: E731
            stage = self._staging[key] = ([mk(t) for t in q], [mk(t) for t in k], [mk(t) for t in v],
                                          [mk(t) for t in out], torch.zeros(n * M + 4 * n + 1, dtype=torch.int32,
                                                                            device=self.dev))
        qd, kd, vd, od, scratch = stage
        ws = self.workspace(n, Hq, M)
        nb = np.ascontiguousarray(n_back, dtype=np.int32)
        if nb.shape != (n,):
            raise ValueError("n_back must hold one count per request")
        vp = ctypes.c_void_p
        pa = self._ptr_array
        stream = torch.cuda.current_stream(self.dev)
        kb._check(kb.lib().kvp_verify_step_device_io(
            self.pages.handle, self.pool.handle, vp(self.table.data_ptr()), self.table.shape[0], self.table.shape[1],
            self.table_mode, vp(rids.data_ptr()), n, M, int(window or 0), int(sinks), Hq, float(scale), pa(q), pa(k),
            pa(v), nb.ctypes.data_as(vp), pa(out), pa(qd), pa(kd), pa(vd), pa(od), vp(scratch.data_ptr()),
            int(self.may_share), vp(ws.data_ptr()), ws.numel(), vp(stream.cuda_stream)), "kvp_verify_step_device_io")

    def check(self):
        """Raise if a device-side error was recorded since the last check."""
        for e, what in ((kb.kvp_sync_error(self.pool), "device"), (self.pages.sync_error(), "device pages")):
            if e != 0:
                raise kb.KvpError(e, what)
