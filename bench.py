#!/usr/bin/env python3
"""Benchmark of the paged decode-attention hot path (one GB300, or N replicas).

One step = one decode step of the whole hot path for every request of the
workload: host bookkeeping (append, copy-on-write, window trim), the device
table write, copy-on-write page copies, store_cache of the new K/V rows and
paged decode attention (work split, attention, split-K combine), for every
layer; the store, the table writes and the attention of a layer are one
launch (store_cache_and_attention), followed by the combine. Prints one
JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

``value`` is the achieved HBM GB/s of the step's algorithmic bytes (K/V rows
attended, q, out, table entries, store_cache rows, table writes and page
copies) with every input already in HBM; ``e2e`` is the same metric through
the public driver (paged_decode_attention_store_gb300.engine) with the
step's q/k/v in pinned host memory, host bookkeeping in the loop and the
output read back each step.
"""

from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")  # the CPU oracle runs on one core

import argparse
import datetime
import json
import math
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_decode_attention_store_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode-attention achieved HBM GB/s (% of GB300 peak); decode tokens/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOADS = ("gqa_decode", "sliding_window", "sliding_window_sinks", "prefix_sharing", "large_batch_p16",
             "large_batch_p1", "gqa_verify4", "gqa_decode_devalloc", "gqa_prefill512")
DEFAULT_WORKLOAD = "large_batch_p16"
# a second workload timed in the same run and reported under "legs"
EXTRA_LEGS = {"large_batch_p16": ("large_batch_p1",)}


# ---------------------------------------------------------------------------
# Workloads as host-operation scripts, replayed by the product and the oracle.
# ---------------------------------------------------------------------------
class Scenario:
    """A workload as a script of host operations. ``layers`` overrides the
    layer count of the 32-layer workloads (a one-layer variant launches the
    same per-layer kernels on the same lengths, for captures that must stay
    small); ``inputs`` is the generator of q/k/v rows (``kv_rows`` and
    ``q_rows`` as in the workloads module, the default)."""

    def __init__(self, name, seed, layers=None, inputs=None, lengths=None):
        self.name = name
        self.seed = seed
        self.inputs = wl if inputs is None else inputs
        self.devalloc = name.endswith("_devalloc")  # page bookkeeping on the device (kvp_dev_*)
        if self.devalloc:
            name = name[:-len("_devalloc")]
        if name == "gqa_decode":
            w = wl.gqa_decode(seed)
        elif name == "sliding_window":
            w = wl.sliding_window(seed)
        elif name == "sliding_window_sinks":
            w = wl.sliding_window_sinks(seed)
        elif name.startswith("gqa_prefill"):
            w = wl.gqa_prefill(seed, chunk=int(name[len("gqa_prefill"):]))
        elif name.startswith("gqa_verify"):
            w = wl.gqa_verify(seed, M=int(name[len("gqa_verify"):]))
        elif name == "prefix_sharing":
            w = wl.prefix_sharing(seed)
        elif name.startswith("large_batch_p"):
            w = wl.large_batch(seed, P=int(name[len("large_batch_p"):]), layers=layers or 32, lengths=lengths)
        else:
            raise ValueError(f"unknown workload {name}")
        self.w = w
        self.ops = []           # prefill script
        self.accumulate = True  # appends touch distinct slots until the first decode step
        if name == "prefix_sharing":
            x = w.extra
            n_req = x["n_prompts"] * x["forks"]
            self.rids = list(range(n_req))
            self.max_requests = n_req + x["n_prompts"]
            for i in range(x["n_prompts"]):
                self.ops.append(("new", n_req + i))
                self.ops.append(("append", n_req + i, x["prompt_len"], 0, 0))
            for f in range(n_req):
                self.ops.append(("fork", n_req + f // x["forks"], f))
            self.ops.append(("batch", list(range(n_req))))  # first suffix token: copy-on-write
            for i in range(x["n_prompts"]):
                self.ops.append(("release", n_req + i))
            for f in range(n_req):
                if x["suffix"][f] > 1:
                    self.ops.append(("append", f, x["suffix"][f] - 1, 0, 0))
            self.lengths = [x["prompt_len"] + s for s in x["suffix"]]
            self.accumulate = False
        else:
            B = len(w.lengths)
            self.rids = list(range(B))
            self.max_requests = B
            self.lengths = list(w.lengths)
            for b, L in enumerate(w.lengths):
                self.ops.append(("new", b))
                if w.window > 0:
                    # the real append + trim path, in chunks of 256 rows; only
                    # rows a later window can reach get data (the sink rows
                    # and the last W - S)
                    t = 0
                    while t < L:
                        n = min(256, L - t)
                        self.ops.append(("append", b, n, max(0, L - (w.window - w.sinks)), w.sinks))
                        t += n
                        self.ops.append(("trim", b, max(0, t + 1 - (w.window - w.sinks)), w.sinks))
                    self.accumulate = False
                else:
                    self.ops.append(("append", b, L, 0, 0))
        self.raw = w.table_mode == "raw"
        # room for the steps' growth: one token a step, or a chunk a step for prefill (72 steps)
        growth = max(512, 72 * w.extra.get("prefill", 0))
        self.max_seq_len = w.extra.get("max_seq_len") if self.raw else max(self.lengths) + growth
        self.window = w.window
        self.sinks = w.sinks
        self.verify = w.extra.get("verify", 0)  # drafted tokens verified per request and step (0: decode)
        self.prefill = w.extra.get("prefill", 0)  # chunk tokens prefilled per request and step (0: decode)
        self.multi = self.verify or self.prefill  # query tokens per request and step, when more than one
        self.l2_resident = name == "prefix_sharing"  # most attended rows are a shared prefix held in L2


def attended_span(sc, L):
    """(se, lo): a step with context L reads rows [0, se) and [lo, L) (for a
    verify step, the union of its M queries' spans)."""
    W, S = sc.w.window, sc.w.sinks
    if W <= 0:
        return 0, 0
    lo = max(0, L - (W + max(sc.multi, 1) - 1 - S))
    se = min(S, lo)
    return (0, 0) if se == lo else (se, lo)


def out_shape(sc):
    """Attention output of one layer: [B, Hq, D], or [B, M, Hq, D] for verify steps."""
    B, w = len(sc.rids), sc.w
    return (B, sc.multi, w.Hq, w.D) if sc.multi else (B, w.Hq, w.D)


def attention_flops(sc, lens):
    """Algorithmic flops of one multi-token attention launch: for every query
    token j (context L - M + j + 1) and query head, 2 D flops per attended key
    for Q K^T and as many for P V (masked work inside tiles not counted)."""
    w, M = sc.w, max(sc.multi, 1)
    keys = 0
    for L in lens:
        for j in range(M):
            Lj = L - M + j + 1
            if w.window > 0:
                lo = max(0, Lj - (w.window - w.sinks))
                se = min(w.sinks, lo)
                keys += (Lj - lo) + (se if se < lo else 0)
            else:
                keys += Lj
    return 4 * w.D * w.Hq * keys


def attended_count(sc, L):
    se, lo = attended_span(sc, L)
    return se + L - lo


def attention_bytes(sc, lens):
    """Algorithmic bytes of one attention launch: attended K/V rows, q, out,
    table entries and context lengths."""
    w = sc.w
    row_kv = 2 * w.Hkv * w.D * (2 if w.dtype == "bf16" else 4)
    elem = 2 if w.dtype == "bf16" else 4
    kv = tab = 0
    for L in lens:
        se, lo = attended_span(sc, L)
        n = se + L - lo
        kv += n * row_kv
        tab += 4 * (n if sc.raw else (-(-se // w.P) + -(-L // w.P) - lo // w.P))
    qo = 2 * len(lens) * max(sc.multi, 1) * w.Hq * w.D * elem
    return kv + qo + tab + 4 * len(lens)


def store_bytes(sc, B):
    """store_cache of one layer: read k and v, write them, read out_loc."""
    w = sc.w
    row = w.Hkv * w.D * (2 if w.dtype == "bf16" else 4)
    return 4 * B * row + 4 * B


def table_write_bytes(sc, n):
    """n (row, col, value) writes: read 12 B, write one entry per page or P per page."""
    return n * (12 + 4 * (sc.w.P if sc.raw else 1))


def step_bytes(sc, lens, n_writes, n_cows, n_trim_writes):
    w = sc.w
    row = w.Hkv * w.D * (2 if w.dtype == "bf16" else 4)
    copies = n_cows * w.layers * 2 * 2 * w.P * row
    return (w.layers * (attention_bytes(sc, lens) + store_bytes(sc, len(lens) * max(sc.multi, 1)))
            + table_write_bytes(sc, n_writes + n_trim_writes) + copies)


def fused_launch_bytes(sc, lens, n_writes, n_cows):
    """Mean algorithmic bytes of one store_cache_and_attention launch of a
    step: the layer's attention and store, and (first layer only, unless the
    step copies pages) the step's table writes."""
    tw = table_write_bytes(sc, n_writes) if n_cows == 0 else 0
    return attention_bytes(sc, lens) + store_bytes(sc, len(lens)) + tw / sc.w.layers


# ---------------------------------------------------------------------------
# GPU arm.
# ---------------------------------------------------------------------------
def _i32(xs, dev):
    return torch.tensor(list(xs), dtype=torch.int32, device=dev)


def device_twin(sc):
    """Whether the workload's e2e leg runs through the device-side page
    bookkeeping (every decode and verify workload; chunked prefill keeps the
    host bookkeeping)."""
    return not sc.devalloc and not sc.prefill


def build_product_device(sc, dev):
    """The scenario's history through the device-side bookkeeping, in the
    order the host replays it: plain histories append every request's rows
    in one call (pages popped in request order); others replay each
    operation (appends, window trims, forks, the first suffix token of a
    batch, releases). The rows are stored layer by layer."""
    from paged_decode_attention_store_gb300.engine import DevicePagedKVCache

    w = sc.w
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    cache = DevicePagedKVCache(w.num_pages, w.P, w.Hkv, w.D, w.layers, w.dtype, max_requests=sc.max_requests,
                               table_mode=w.table_mode, max_seq_len=sc.max_seq_len, free_stack=w.free_order,
                               device=dev)
    pend = []  # (rids, positions, slots) waiting to be stored

    def flush():
        if not pend:
            return
        rr = torch.cat([p[0] for p in pend])
        pos = torch.cat([p[1] for p in pend])
        slots = torch.cat([p[2] for p in pend])
        step = 1 << 18
        for layer in range(w.layers):
            for s0 in range(0, rr.numel(), step):
                k, v = sc.inputs.kv_rows(sc.seed, layer, rr[s0:s0 + step], pos[s0:s0 + step], w.Hkv, w.D, dtype=tdt,
                                         device=dev)
                cache.store(layer, k, v, slots[s0:s0 + step].contiguous())
        pend.clear()

    def add_store(rid_list, pos_list, slots):
        pend.append((torch.as_tensor(rid_list, dtype=torch.int64, device=dev),
                     torch.as_tensor(pos_list, dtype=torch.int64, device=dev), slots))

    plain = all(op[0] == "new" or (op[0] == "append" and not op[3] and not op[4]) for op in sc.ops)
    lengths = {}
    if plain:
        rids = [op[1] for op in sc.ops if op[0] == "new"]
        counts = {op[1]: op[2] for op in sc.ops if op[0] == "append"}
        cache.new(rids)
        cnt = [counts.get(r, 0) for r in rids]
        slots = cache.append(rids, counts=cnt)
        add_store([r for r, c in zip(rids, cnt) for _ in range(c)], [t for c in cnt for t in range(c)], slots)
        lengths = dict(zip(rids, cnt))
    else:
        for op in sc.ops:
            kind = op[0]
            if kind == "new":
                cache.new([op[1]])
                lengths[op[1]] = 0
            elif kind == "append":
                _, rid, n, store_from, store_below = op
                L0 = lengths[rid]
                slots = cache.append([rid], counts=[n])
                lengths[rid] = L0 + n
                first = max(store_from, L0)
                if first < L0 + n:
                    add_store([rid] * (L0 + n - first), list(range(first, L0 + n)), slots[first - L0:])
                sink_end = min(store_below, first, L0 + n)
                if L0 < sink_end:
                    add_store([rid] * (sink_end - L0), list(range(L0, sink_end)), slots[:sink_end - L0])
            elif kind == "batch":
                flush()
                slots = cache.append(op[1])
                add_store(op[1], [lengths[r] for r in op[1]], slots)
                for r in op[1]:
                    lengths[r] += 1
            elif kind == "trim":
                cache.pages.trim(cache._i32([op[1]]), keep_from=cache._i32([op[2]]), sinks=op[3])
            elif kind == "fork":
                flush()
                cache.fork([op[1]], [op[2]])
                lengths[op[2]] = lengths[op[1]]
            elif kind == "release":
                cache.release([op[1]])
                del lengths[op[1]]
            if not sc.accumulate:
                flush()
    flush()
    torch.cuda.synchronize(dev)
    cache.check()
    return cache, [lengths[r] for r in sc.rids]


def build_product(sc, dev):
    from paged_decode_attention_store_gb300.engine import PagedKVCache

    w = sc.w
    if sc.devalloc:
        return build_product_device(sc, dev)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    cache = PagedKVCache(w.num_pages, w.P, w.Hkv, w.D, w.layers, w.dtype, max_requests=sc.max_requests,
                         table_mode=w.table_mode, max_seq_len=sc.max_seq_len, free_stack=w.free_order, device=dev)
    lengths = {}
    pend = []  # (rids, positions, slots) waiting to be stored

    def flush():
        if not pend:
            return
        rids = torch.cat([p[0] for p in pend])
        pos = torch.cat([p[1] for p in pend])
        slots = torch.cat([p[2] for p in pend])
        step = 1 << 18
        for layer in range(w.layers):
            for s in range(0, rids.numel(), step):
                k, v = sc.inputs.kv_rows(sc.seed, layer, rids[s:s + step], pos[s:s + step], w.Hkv, w.D, dtype=tdt,
                                  device=dev)
                cache.store(layer, k, v, slots[s:s + step].contiguous())
        pend.clear()

    def add_store(rid_list, pos_list, slots):
        pend.append((torch.as_tensor(rid_list, dtype=torch.int64, device=dev),
                     torch.as_tensor(pos_list, dtype=torch.int64, device=dev), slots))

    for op in sc.ops:
        kind = op[0]
        if kind == "new":
            cache.new(op[1])
            lengths[op[1]] = 0
        elif kind == "append":
            _, rid, n, store_from, store_below = op
            L0 = lengths[rid]
            slots = cache.append([rid] * n)
            lengths[rid] = L0 + n
            first = max(store_from, L0)
            if first < L0 + n:
                add_store([rid] * (L0 + n - first), list(range(first, L0 + n)), slots[first - L0:])
            sink_end = min(store_below, first, L0 + n)  # sink rows below the stored tail
            if L0 < sink_end:
                add_store([rid] * (sink_end - L0), list(range(L0, sink_end)), slots[:sink_end - L0])
        elif kind == "batch":
            rids = op[1]
            flush()
            slots = cache.append(rids)
            add_store(rids, [lengths[r] for r in rids], slots)
            for r in rids:
                lengths[r] += 1
        elif kind == "trim":
            cache.trim(op[1], op[2], sinks=op[3])
        elif kind == "fork":
            flush()
            cache.fork(op[1], op[2])
            lengths[op[2]] = lengths[op[1]]
        elif kind == "release":
            cache.release(op[1])
            del lengths[op[1]]
        if not sc.accumulate:
            flush()
    flush()
    torch.cuda.synchronize(dev)
    cache.check()
    return cache, [lengths[r] for r in sc.rids]


class StepData:
    """Host decisions and device inputs of one decode step, prepared up front."""


def prepare_steps(sc, cache, lens, first_step, n_steps, dev, host_inputs=False):
    w = sc.w
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    steps = []
    lens = list(lens)
    for s in range(first_step, first_step + n_steps):
        if sc.devalloc:
            st, lens = _prepare_device_step(sc, lens, s, dev, host_inputs)
            steps.append(st)
            continue
        if sc.multi:
            st, lens = _prepare_verify_step(sc, cache, lens, s, dev, host_inputs)
            steps.append(st)
            continue
        st = StepData()
        slots, writes, cows = cache.host.append(sc.rids)
        np.add.at(cache.lengths, np.asarray(sc.rids, np.int64), 1)
        st.n_writes, st.n_cows = len(writes), len(cows)
        st.pre = None if not writes else tuple(_i32(x, dev) for x in zip(*writes))
        st.cows = None if not cows else tuple(_i32(x, dev) for x in zip(*cows))
        st.out_loc = _i32(slots, dev)
        positions = list(lens)
        lens = [L + 1 for L in lens]
        st.lens_list = list(lens)
        st.lens = _i32(lens, dev)
        post = []
        if sc.window > 0:
            for r, L in zip(sc.rids, lens):
                post += cache.host.trim(r, max(0, L + 1 - (sc.window - sc.sinks)), sinks=sc.sinks)
        st.n_post = len(post)
        st.post = None if not post else tuple(_i32(x, dev) for x in zip(*post))
        st.q, st.k, st.v = [], [], []
        for layer in range(w.layers):
            q = sc.inputs.q_rows(sc.seed, s, layer, sc.rids, w.Hq, w.D, dtype=tdt, device=dev)
            k, v = sc.inputs.kv_rows(sc.seed, layer, sc.rids, positions, w.Hkv, w.D, dtype=tdt, device=dev)
            if host_inputs:
                q, k, v = (x.cpu().pin_memory() for x in (q, k, v))
            st.q.append(q)
            st.k.append(k)
            st.v.append(v)
        st.bytes = step_bytes(sc, lens, st.n_writes, st.n_cows, st.n_post)
        st.attn_bytes = fused_launch_bytes(sc, lens, st.n_writes, st.n_cows)
        steps.append(st)
    return steps, lens


def _prepare_device_step(sc, lens, s, dev, host_inputs):
    """A decode step whose bookkeeping runs on the device: only q/k/v are
    prepared (no host decision); the step's table writes are counted from
    the lengths (a new page on every page boundary)."""
    w = sc.w
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    st = StepData()
    st.rids = _i32(sc.rids, dev)
    st.n_writes = sum(1 for L in lens if L % w.P == 0)
    st.n_cows = st.n_post = 0
    st.pre = st.cows = st.post = None
    positions = list(lens)
    lens = [L + 1 for L in lens]
    st.lens_list = list(lens)
    st.q, st.k, st.v = [], [], []
    for layer in range(w.layers):
        q = sc.inputs.q_rows(sc.seed, s, layer, sc.rids, w.Hq, w.D, dtype=tdt, device=dev)
        k, v = sc.inputs.kv_rows(sc.seed, layer, sc.rids, positions, w.Hkv, w.D, dtype=tdt, device=dev)
        if host_inputs:
            q, k, v = (x.cpu().pin_memory() for x in (q, k, v))
        st.q.append(q)
        st.k.append(k)
        st.v.append(v)
    st.bytes = step_bytes(sc, lens, st.n_writes, 0, 0)
    st.attn_bytes = fused_launch_bytes(sc, lens, st.n_writes, 0)
    return st, lens


def _prepare_verify_step(sc, cache, lens, s, dev, host_inputs):
    """A multi-token step: M tokens per request appended and stored, then
    attended at once. A speculative (verify) step then accepts a seeded
    number of the M drafts and rewinds the rest; a prefill step keeps all."""
    w, M = sc.w, sc.multi
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    st = StepData()
    rr = [r for r in sc.rids for _ in range(M)]
    slots, writes, cows = cache.host.append(rr)
    np.add.at(cache.lengths, np.asarray(rr, np.int64), 1)
    st.n_writes, st.n_cows = len(writes), len(cows)
    st.pre = None if not writes else tuple(_i32(x, dev) for x in zip(*writes))
    st.cows = None if not cows else tuple(_i32(x, dev) for x in zip(*cows))
    st.out_loc = _i32(slots, dev)
    positions = [L + j for L in lens for j in range(M)]
    ctx = [L + M for L in lens]
    st.lens_list = list(ctx)
    st.lens = _i32(ctx, dev)
    acc = wl.accepted_drafts(sc.seed, s, len(sc.rids), M) if sc.verify else [M] * len(sc.rids)
    post = []
    for r, a in zip(sc.rids, acc):
        if a < M:
            post += cache.host.rewind(r, M - a)
            cache.lengths[r] -= M - a
    st.n_post = len(post)
    st.post = None if not post else tuple(_i32(x, dev) for x in zip(*post))
    st.q, st.k, st.v = [], [], []
    for layer in range(w.layers):
        q = torch.stack([sc.inputs.q_rows(sc.seed, s * M + j, layer, sc.rids, w.Hq, w.D, dtype=tdt, device=dev)
                         for j in range(M)], dim=1).contiguous()
        k, v = sc.inputs.kv_rows(sc.seed, layer, rr, positions, w.Hkv, w.D, dtype=tdt, device=dev)
        if host_inputs:
            q, k, v = (x.cpu().pin_memory() for x in (q, k, v))
        st.q.append(q)
        st.k.append(k)
        st.v.append(v)
    st.bytes = step_bytes(sc, ctx, st.n_writes, st.n_cows, st.n_post)
    st.attn_bytes = attention_bytes(sc, ctx)
    st.attn_flops = attention_flops(sc, ctx)
    st.accepted = sum(acc)
    return st, [L + a for L, a in zip(lens, acc)]


def run_step(sc, cache, st, outs, events=None):
    """Issue one prepared step; returns the number of kernels launched.

    Copy-on-write pages first (with the step's table writes when there are
    copies: a copied tail page's entry is read by the attention), then one
    store_cache_and_attention launch per layer, the first carrying the
    step's new-page table writes; last the window's releases."""
    from paged_decode_attention_store_gb300 import binding as kb

    w = sc.w
    P = w.P
    n = 0
    if sc.devalloc:  # device append, fused store + attention (+ combine) per layer, device trim
        if events is not None:
            kb.kvp_pool_set_timing_events(cache.pool, *events.pop())
        cache.decode_step(st.rids, st.q, st.k, st.v, outs, sc.window, w.scale, sinks=sc.sinks)
        return 1 + 2 * w.layers + (1 if sc.window > 0 else 0) + (1 if cache.may_share else 0)
    if sc.multi:  # table writes, store of the M rows, verify (+ combine) or prefill, rewind writes
        if st.pre is not None:
            kb.page_table_write(cache.table, *st.pre, expand=P if sc.raw else 1, error_word=cache.pool.error_word)
            n += 1
        if st.cows is not None:
            kb.copy_pages(cache.pool, *st.cows)
            n += 1
        for layer in range(w.layers):
            cache.store(layer, st.k[layer], st.v[layer], st.out_loc)
            if events is not None:
                kb.kvp_pool_set_timing_events(cache.pool, *events.pop())
            if sc.verify:
                cache.verify(layer, st.q[layer], st.lens, sc.window, w.scale, outs[layer], sinks=sc.sinks)
                n += 3
            else:
                cache.prefill(layer, st.q[layer], st.lens, sc.window, w.scale, outs[layer], sinks=sc.sinks)
                n += 2
        if st.post is not None:
            kb.page_table_write(cache.table, *st.post, expand=P if sc.raw else 1, error_word=cache.pool.error_word)
            n += 1
        return n
    pre = st.pre
    if st.cows is not None:
        kb.copy_pages(cache.pool, *st.cows)
        n += 1
        if pre is not None:
            kb.page_table_write(cache.table, *pre, expand=P if sc.raw else 1, error_word=cache.pool.error_word)
            n += 1
            pre = None
    fused = w.dtype == "bf16" and w.D == 128  # one launch; else table write, store and the general kernel
    for layer in range(w.layers):
        if events is not None:
            kb.kvp_pool_set_timing_events(cache.pool, *events.pop())
        tw = pre if layer == 0 else None
        cache.store_and_attend(layer, st.q[layer], st.k[layer], st.v[layer], st.out_loc, st.lens, sc.window,
                               w.scale, outs[layer], table_writes=tw, sinks=sc.sinks)
        n += 2 if fused else 2 + (tw is not None)  # fused kernel + combine, or write, store, general kernel
    if st.post is not None:
        kb.page_table_write(cache.table, *st.post, expand=P if sc.raw else 1, error_word=cache.pool.error_word)
        n += 1
    return n


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            uuid = str(torch.cuda.get_device_properties(dev_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(dev_index)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        self.file.close()
        os.unlink(self.file.name)
        inside = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "reasons": reasons, "samples": len(inside)}


def measured_peak(key="hbm_gbs", fallback=None):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except (OSError, KeyError, ValueError):
        return (FALLBACK_HBM_GBS if fallback is None else fallback), "fallback"


def ncu_summary(kernel, source, workload):
    """The ``key: value`` lines of the committed ncu summary of ``kernel`` on
    ``workload``, if it was taken on the current source of that kernel."""
    import hashlib

    src = os.path.join(ROOT, "paged_decode_attention_store_gb300", "csrc", source)
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        vals = {}
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    except OSError:
        return None
    return vals if vals.get("kernel_source_sha256_16") == digest else None


def ncu_traffic(workload):
    """DRAM bytes per launch of the decode attention kernel from its ncu summary."""
    vals = ncu_summary("tc_decode_kernel", "attention_tc.cu", workload)
    try:
        return float(vals["dram_bytes_per_launch"]) if vals else None
    except (KeyError, ValueError):
        return None


def ncu_prefill_traffic(workload, flops):
    """DRAM bytes of a prefill launch of ``flops`` algorithmic flops: the
    captured launch's bytes scaled by flops (both grow with the tiles' key
    counts; the L2 hit rate falls as contexts grow, so this is a lower bound)."""
    vals = ncu_summary("prefill_tc_kernel", "prefill_tc.cu", workload)
    try:
        return round(float(vals["dram_bytes_per_launch"]) * flops / float(vals["algorithmic_flops_per_launch"]))
    except (TypeError, KeyError, ValueError, ZeroDivisionError):
        return None


def reduce_over_ranks(elapsed_ms, total_bytes, tokens, e2e_ms, e2e_bytes, world, device):
    """Whole-job totals: the slowest rank's times, every rank's bytes and tokens."""
    if world <= 1:
        return elapsed_ms, total_bytes, tokens, e2e_ms, e2e_bytes
    stats = torch.tensor([elapsed_ms, total_bytes, tokens, e2e_ms, e2e_bytes], dtype=torch.float64, device=device)
    mx = stats.clone()
    torch.distributed.all_reduce(mx, op=torch.distributed.ReduceOp.MAX)
    sm = stats.clone()
    torch.distributed.all_reduce(sm, op=torch.distributed.ReduceOp.SUM)
    return mx[0].item(), sm[1].item(), sm[2].item(), mx[3].item(), sm[4].item()


def run_gpu(args, rank, world, local_rank):
    """The headline workload's line, with the extra legs of the same run
    (each timed the same way, one after the other) under ``legs``."""
    line = measure(args, args.workload, rank, world, local_rank, with_cpu=True)
    if args.no_extra:
        return line
    for name in EXTRA_LEGS.get(args.workload, ()):
        gc_cuda()
        leg = measure(args, name, rank, world, local_rank, with_cpu=False)
        if line is not None:
            line.setdefault("legs", {})[name] = {k: leg[k] for k in (
                "value", "unit", "ms_per_step", "tokens_per_s", "pct_of_peak", "pct_of_nominal_8tbs", "gpu_launches",
                "roofline", "e2e", "clocks", "config")}
    return line


def gc_cuda():
    import gc

    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def measure(args, name, rank, world, local_rank, with_cpu):
    from paged_decode_attention_store_gb300 import binding as kb
    from paged_decode_attention_store_gb300.engine import PagedKVCache  # noqa: F401  (fail loudly if missing)

    kb.lib()
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    sc = Scenario(name, args.seed + rank, layers=args.layers)
    w = sc.w
    cache, lens = build_product(sc, dev)
    K, W = args.steps, args.warmup
    # W warm-up steps, K timed steps for `value` (nothing between the kernels
    # but the step's own launches), then K more steps with events around each
    # attention kernel for the roofline (an event between two kernels stops
    # the second from launching early, so it is kept out of the first pass).
    steps, lens_after = prepare_steps(sc, cache, lens, 1, W + 2 * K, dev)
    tdt = cache.tdt
    outs = [torch.empty(out_shape(sc), dtype=tdt, device=dev) for _ in range(w.layers)]
    soak_out = torch.empty((len(sc.rids), w.Hq, w.D), dtype=tdt, device=dev)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    # soak: repeat the current state's attention ~1 s so clocks settle and get
    # sampled. The history was trimmed for the first decode step (context
    # L + 1), so at context L the window is one row shorter.
    t_soak = time.time()
    soak_window = sc.window - 1 if sc.window > 0 else 0
    while time.time() - t_soak < args.soak:
        for layer in range(w.layers):
            q0 = steps[0].q[layer][:, 0].contiguous() if sc.multi else steps[0].q[layer]
            cache.attend(layer, q0, _i32(lens, dev), soak_window, w.scale, soak_out, sinks=sc.sinks)
        torch.cuda.synchronize(dev)
    for i in range(W):
        run_step(sc, cache, steps[i], outs)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    t0 = time.time()
    start.record()
    for i in range(W, W + K):
        launches += run_step(sc, cache, steps[i], outs)
    end.record()
    torch.cuda.synchronize(dev)
    t1 = time.time()
    elapsed_ms = start.elapsed_time(end)
    if world > 1:
        torch.distributed.barrier()

    n_attn = K if sc.devalloc else K * w.layers  # the native device step times its first layer
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_attn)]
    for a, b in ev_pairs:  # torch creates the CUDA event at its first record
        a.record()
        b.record()
    torch.cuda.synchronize(dev)
    pending = list(reversed(ev_pairs))
    for i in range(W + K, W + 2 * K):
        run_step(sc, cache, steps[i], outs, events=pending)
    torch.cuda.synchronize(dev)
    # the clock record covers the device-timed region; nvidia-smi's polling
    # is stopped before the end-to-end leg, whose per-step host
    # synchronisation it would otherwise slow down
    clocks = sampler.stop(t0, t1) if sampler else None
    cache.check()
    attn_ms = [a.elapsed_time(b) for a, b in ev_pairs]
    total_bytes = sum(st.bytes for st in steps[W:W + K])
    # tokens a step adds: one per request, or the accepted drafts of a verify step
    timed_tokens = sum(st.accepted for st in steps[W:W + K]) if sc.multi else K * len(sc.rids)
    attn_bytes_mean = statistics.mean(st.attn_bytes for st in steps[W + K:W + 2 * K])

    # end to end through the public API, host buffers: the device-side page
    # bookkeeping (no host decision per step) when the history is plain,
    # else the host bookkeeping's native step
    if device_twin(sc):
        del cache
        torch.cuda.empty_cache()
        sc_dev = Scenario(sc.name + "_devalloc", sc.seed, layers=args.layers)
        cache, lens_dev = build_product_device(sc_dev, dev)
        e2e = run_e2e(args, sc_dev, cache, lens_dev, W + 2 * K + 1, dev)
        e2e["path"] = ("DevicePagedKVCache.verify_step_host (kvp_verify_step_device_io: drafts appended, stored, "
                       "verified and the rejected ones rewound with the page bookkeeping on the device, host copies "
                       "in the same native call)" if sc.verify else
                       "DevicePagedKVCache.decode_step_host (kvp_decode_step_device_io: page bookkeeping, window "
                       "trim included, on the device, host copies in the same native call)")
    else:
        e2e = run_e2e(args, sc, cache, lens_after, W + 2 * K + 1, dev)
        e2e["path"] = ("DevicePagedKVCache.decode_step" if sc.devalloc else
                       "PagedKVCache.verify_step + rewind" if sc.verify else
                       "PagedKVCache.prefill_step" if sc.prefill else
                       "PagedKVCache.decode_step (kvp_decode_step: host page bookkeeping)")

    elapsed_ms, total_bytes, tokens, e2e_ms, e2e_bytes = reduce_over_ranks(
        elapsed_ms, float(total_bytes), float(timed_tokens), e2e["ms"], float(e2e["bytes"]), world, dev)
    if rank != 0:
        return None

    peak, peak_kind = measured_peak()
    value = total_bytes / (elapsed_ms * 1e-3) / 1e9
    achieved = attn_bytes_mean / (statistics.mean(attn_ms) * 1e-3) / 1e9
    traffic = ncu_traffic(sc.name)
    launch_s = statistics.mean(attn_ms) * 1e-3
    roofline = {
        "bound": "hbm",
        "kernel": "tc_decode_kernel",
        "achieved": round(achieved, 1),
        "peak": peak,
        "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)",
        "unit": "GB/s",
        "frac": round(achieved / peak, 4),
        "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
        "traffic": traffic,
        "basis": "algorithmic bytes per launch / CUDA-event launch time",
        "dram_gbs": None if traffic is None else round(traffic / launch_s / 1e9, 1),
        "algorithmic_bytes_per_launch": int(attn_bytes_mean),
        "mean_launch_us": round(1e3 * statistics.mean(attn_ms), 2),
        "launches_timed": len(attn_ms),
    }
    if sc.l2_resident:
        # most of the logical bytes are the shared prefix, served from L2: the
        # fraction of the HBM peak is taken on the DRAM bytes ncu counted for
        # one launch of this workload, the logical rate reported beside it
        dram = None if traffic is None else traffic / launch_s / 1e9
        roofline.update({
            "achieved": None if dram is None else round(dram, 1),
            "frac": None if dram is None else round(dram / peak, 4),
            "frac_of_nominal_8tbs": None if dram is None else round(dram / NOMINAL_HBM_GBS, 4),
            "logical_gbs": round(achieved, 1),
            "basis": ("ncu DRAM bytes per launch (dram__bytes_read + write) / CUDA-event launch time" if dram is not None
                      else "no ncu summary of the current kernel source: DRAM bytes unknown (logical bytes are "
                           "mostly L2 hits and would overstate the HBM rate)"),
        })
    if sc.prefill:  # a dense contraction: flops against the measured bf16 tensor peak
        flops_mean = statistics.mean(st.attn_flops for st in steps[W + K:W + 2 * K])
        tf = flops_mean / (statistics.mean(attn_ms) * 1e-3) / 1e12
        tpeak, tkind = measured_peak("bf16_tflops", 1900.0)
        roofline.update({"bound": "tensor", "kernel": "prefill_tc_kernel", "achieved": round(tf, 1), "peak": tpeak,
                         "peak_kind": f"{tkind} bf16_tflops (cuBLAS, burst)", "unit": "TFLOP/s",
                         "frac": round(tf / tpeak, 4), "frac_of_nominal_8tbs": None,
                         "traffic": ncu_prefill_traffic(sc.name, flops_mean),
                         "algorithmic_flops_per_launch": int(flops_mean), "attention_gbps": round(achieved, 1)})
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(elapsed_ms / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded counter-based generator; lengths from the workload's distribution)",
        "config": {
            "workload": sc.name,
            "batch": len(sc.rids),
            "q_heads": w.Hq,
            "kv_heads": w.Hkv,
            "head_dim": w.D,
            "page_size": w.P,
            "layers": w.layers,
            "window": w.window,
            "sinks": w.sinks,
            "verify_tokens": sc.verify,
            "prefill_chunk": sc.prefill,
            "table": "raw token locations" if sc.raw else "block table",
            "mean_attended_tokens": round(statistics.mean(
                attended_count(sc, L) for L in steps[W].lens_list), 1),
            "kv_bytes_per_step": int(sum(attended_count(sc, L) for L in steps[W].lens_list)
                                     * 2 * w.Hkv * w.D * 2 * w.layers),
            "l2": ("no flush: the shared prefix (8 x 129 pages, 67.6 MB) stays L2-resident by design; roofline.frac "
                   "uses ncu DRAM bytes" if sc.l2_resident else
                   "no flush: inputs larger than L2 (K/V read per step >> 129 MB)"),
            "seed": args.seed,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "tokens_per_s": round(tokens / (elapsed_ms * 1e-3), 1),
        "pct_of_peak": round(100.0 * value / peak, 2),
        "pct_of_nominal_8tbs": round(100.0 * value / NOMINAL_HBM_GBS, 2),
        "gpu_launches": launches,
        "roofline": roofline,
        "e2e": {
            "value": round(e2e_bytes / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": UNIT,
            "tokens_per_s": round(tokens / (e2e_ms * 1e-3), 1),
            "ms_per_step": round(e2e_ms / K, 4),
            "h2d_bytes_per_step": e2e["h2d"],
            "d2h_bytes_per_step": e2e["d2h"],
            "host_link": e2e["link"],
            "pinned_input_sets": e2e["input_sets"],
            "warmup_steps": e2e["warmup"],
            "path": e2e["path"],
        },
        "clocks": clocks,
    }
    if world == 1 and with_cpu and not args.no_cpu_baseline:
        single = cpu_baseline(sc, args.cpu_seconds)
        line["cpu_baseline"] = single
        try:
            allc = cpu_baseline_all_cores(sc, args.cpu_seconds, min(os.cpu_count() or 1, 16))
            line["cpu_baseline"] = dict(single, value=allc["value"], cores=allc["cores"], sample=allc["sample"],
                                        single_core={"value": single["value"], "sample": single["sample"]})
        except Exception as e:  # keep the single-core figure, and say why
            line["cpu_baseline"]["all_cores_unavailable"] = repr(e)[:200]
    return line


E2E_INPUT_SETS = 4  # distinct pinned input sets the end-to-end leg cycles through


def run_e2e(args, sc, cache, lens, first_step, dev):
    """W untimed and K timed steps through the public driver with pinned
    host q/k/v and outputs: bookkeeping, all copies and the output read-back
    (each call returns once the step's output is on the host) are inside the
    timing. The steps cycle through E2E_INPUT_SETS distinct pinned input sets,
    as a caller reuses its staging buffers (one pinned set per step of a long
    run would make the copies slower as the GPU's translation of host memory
    runs out: a step over 20 distinct 160 MB sets took 15-29 ms against 8.8 ms
    over a reused few)."""
    w = sc.w
    K, W = args.steps, args.warmup
    R = min(K + W, E2E_INPUT_SETS)
    host_sets = _host_inputs(sc, first_step, R, lens)
    out_host = _pinned(shapes=[out_shape(sc)] * w.layers, dtype=cache.tdt)
    if sc.devalloc:
        return _run_e2e_device(sc, cache, lens, host_sets, out_host, dev, first_step, K, W)
    rids = np.asarray(sc.rids, np.int32)

    def step(s):
        """One step; returns what its bytes are computed from (after the timing)."""
        q_h, k_h, v_h = host_sets[s % R]
        if sc.prefill:  # a chunk per request: append, store, attend
            cache.prefill_step(rids, q_h, k_h, v_h, out_host, sc.window, w.scale, sinks=sc.sinks)
            return cache.lengths[rids].copy(), cache.last_writes, cache.last_copies, 0
        if sc.verify:  # draft M, verify, accept the seeded count, rewind the rest
            M = sc.verify
            cache.verify_step(rids, q_h, k_h, v_h, out_host, sc.window, w.scale, sinks=sc.sinks)
            ctx = cache.lengths[rids].copy()
            n_writes, n_cows = cache.last_writes, cache.last_copies
            n_back = 0
            for r, a in zip(sc.rids, wl.accepted_drafts(sc.seed, first_step + s, len(sc.rids), M)):
                n_back += cache.rewind(r, M - a)
            return ctx, n_writes, n_cows, n_back
        cache.decode_step(rids, q_h, k_h, v_h, out_host, sc.window, w.scale, sinks=sc.sinks)
        return cache.lengths[rids].copy(), cache.last_writes, cache.last_copies, cache.last_trims

    for s in range(W):
        step(s)
    torch.cuda.synchronize(dev)
    cache.h2d_bytes = 0
    records = []
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for s in range(W, W + K):
        records.append(step(s))
    end.record()
    torch.cuda.synchronize(dev)
    total_bytes = sum(step_bytes(sc, [int(x) for x in lens_], nw, nc, nt) for lens_, nw, nc, nt in records)
    cache.check()
    d2h = sum(o.numel() * o.element_size() for o in out_host)
    return {"ms": start.elapsed_time(end), "bytes": total_bytes, "h2d": cache.h2d_bytes // K, "d2h": d2h,
            "link": link_rates(dev), "input_sets": R, "warmup": W}


def _run_e2e_device(sc, cache, lens, host_sets, out_host, dev, first_step, K, W):
    """End to end with the bookkeeping on the device: per step one native
    call copies q/k/v in from pinned host memory, runs the step (a decode
    step, or a verify step that rewinds the rejected drafts) and copies the
    output back; no host decision, no table writes from the host. The step's
    table writes are counted for the bytes from the lengths. W untimed steps
    first, then K timed ones."""
    w = sc.w
    R = len(host_sets)
    P = w.P
    rids = torch.as_tensor(sc.rids, dtype=torch.int32, device=dev)
    lens = list(lens)
    M = max(sc.verify, 1)

    # every step's inputs and byte count are known before the timing starts
    backs, step_b = [], []
    for s in range(W + K):
        if sc.verify:
            back = [M - a for a in wl.accepted_drafts(sc.seed, first_step + s, len(sc.rids), M)]
            ctx = [L + M for L in lens]
            n_writes = sum(-(-c // P) - -(-L // P) for L, c in zip(lens, ctx))
            after = [c - nb for c, nb in zip(ctx, back)]
            n_back = sum(-(-c // P) - -(-a // P) for c, a in zip(ctx, after))
            backs.append(back)
            step_b.append(step_bytes(sc, ctx, n_writes, 0, n_back))
            lens = after
            continue
        n_writes = sum(1 for L in lens if L % P == 0)
        lens = [L + 1 for L in lens]
        n_trim = 0
        if sc.window > 0:  # pages the step's trim releases: those that fall wholly below L + 1 - (W - S)
            kf = lambda L: max(0, L + 1 - (sc.window - sc.sinks)) // P  # noqa: E731
            n_trim = sum(max(0, kf(L) - kf(L - 1)) for L in lens)
        step_b.append(step_bytes(sc, lens, n_writes, 0, n_trim))

    def step(s):
        q_h, k_h, v_h = host_sets[s % R]
        if sc.verify:
            cache.verify_step_host(rids, q_h, k_h, v_h, backs[s], out_host, sc.window, w.scale, sinks=sc.sinks)
        else:
            cache.decode_step_host(rids, q_h, k_h, v_h, out_host, sc.window, w.scale, sinks=sc.sinks)

    for s in range(W):
        step(s)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for s in range(W, W + K):
        step(s)
    end.record()
    torch.cuda.synchronize(dev)
    total_bytes = sum(step_b[W:])
    cache.check()
    h2d = sum(x[i].numel() * x[i].element_size() for x in host_sets[0] for i in range(w.layers))
    d2h = sum(o.numel() * o.element_size() for o in out_host)
    return {"ms": start.elapsed_time(end), "bytes": total_bytes, "h2d": h2d + (4 * len(sc.rids) if sc.verify else 0),
            "d2h": d2h, "link": link_rates(dev), "input_sets": R, "warmup": W}


def link_rates(dev, nbytes=128 << 20):
    """Host<->device copy rates of this machine (pinned memory), GB/s."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d_gbs", d, h), ("d2h_gbs", h, d)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize(dev)
        out[name] = round(3 * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
    return out


def _pinned(tensors=None, shapes=None, dtype=None):
    """Views into ONE pinned host buffer (each 256-byte aligned): copies of
    ``tensors``, or empty tensors of ``shapes`` and ``dtype``. The copy engines
    reach pinned memory through the GPU's translation of host addresses; one
    contiguous region per step's inputs (and one for the outputs) keeps that
    translation compact, where hundreds of separate pinned tensors made the
    end-to-end step time swing by a fifth from run to run."""
    if tensors is not None:
        shapes, dtypes = [t.shape for t in tensors], [t.dtype for t in tensors]
    else:
        dtypes = [dtype] * len(shapes)
    nbytes = [int(np.prod(sh)) * torch.empty((), dtype=dt).element_size() for sh, dt in zip(shapes, dtypes)]
    buf = torch.empty(sum((n + 255) // 256 * 256 for n in nbytes), dtype=torch.uint8, pin_memory=True)
    views, off = [], 0
    for i, (sh, dt, n) in enumerate(zip(shapes, dtypes, nbytes)):
        v = buf[off:off + n].view(dt).view(sh)
        if tensors is not None:
            v.copy_(tensors[i])
        views.append(v)
        off += (n + 255) // 256 * 256
    return views


def _host_inputs(sc, first_step, K, lens):
    """Pinned host copies of each step's q, k, v (generated on the device),
    one pinned buffer per step."""
    w = sc.w
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = torch.device("cuda", torch.cuda.current_device())
    out = []
    if sc.multi:
        M = sc.multi
        lens = list(lens)
        rr = [r for r in sc.rids for _ in range(M)]
        for s in range(first_step, first_step + K):
            positions = [L + j for L in lens for j in range(M)]
            qs, ks, vs = [], [], []
            for layer in range(w.layers):
                q = torch.stack([sc.inputs.q_rows(sc.seed, s * M + j, layer, sc.rids, w.Hq, w.D, dtype=tdt, device=dev)
                                 for j in range(M)], dim=1)
                k, v = sc.inputs.kv_rows(sc.seed, layer, rr, positions, w.Hkv, w.D, dtype=tdt, device=dev)
                qs.append(q)
                ks.append(k)
                vs.append(v)
            h = _pinned(qs + ks + vs)
            L_ = w.layers
            out.append((h[:L_], h[L_:2 * L_], h[2 * L_:]))
            acc = wl.accepted_drafts(sc.seed, s, len(sc.rids), M) if sc.verify else [M] * len(sc.rids)
            lens = [L + a for L, a in zip(lens, acc)]
        return out
    for i, s in enumerate(range(first_step, first_step + K)):
        positions = [L + i for L in lens]
        qs, ks, vs = [], [], []
        for layer in range(w.layers):
            q = sc.inputs.q_rows(sc.seed, s, layer, sc.rids, w.Hq, w.D, dtype=tdt, device=dev)
            k, v = sc.inputs.kv_rows(sc.seed, layer, sc.rids, positions, w.Hkv, w.D, dtype=tdt, device=dev)
            qs.append(q)
            ks.append(k)
            vs.append(v)
        h = _pinned(qs + ks + vs)
        L_ = w.layers
        out.append((h[:L_], h[L_:2 * L_], h[2 * L_:]))
    return out


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and --impl reference).
# ---------------------------------------------------------------------------
class OracleSample:
    """The oracle replaying the scenario's script, storing rows of ``track`` only."""

    def __init__(self, sc, track, layers=None):
        import oracle.attention as OA
        from oracle.pagetable import PageTable
        from oracle.raw_locations import RawLocationTable

        self.OA = OA
        self.sc, w = sc, sc.w
        self.track = set(track)
        self.pt = PageTable(w.num_pages, w.P, free_order=w.free_order)
        self.raw = None
        if sc.raw:
            self.raw = RawLocationTable(w.num_pages, w.P, sc.max_requests, sc.max_seq_len,
                                        free_page_order=w.free_order)
        self.stores = [OA.SlotStore() for _ in range(w.layers)]
        self.layers = list(range(w.layers)) if layers is None else list(layers)
        self.tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        for op in sc.ops:
            self._op(op)

    def _store(self, rid, positions, slots):
        if rid not in self.track or not positions:
            return
        w = self.sc.w
        for layer in self.layers:
            k, v = self.sc.inputs.kv_rows(self.sc.seed, layer, rid, positions, w.Hkv, w.D, dtype=self.tdt)
            self.stores[layer].store_cache(slots, k.float().numpy(), v.float().numpy())

    def _append(self, rids):
        before = {}
        for r in rids:
            before.setdefault(r, self.pt.length[r])
        res = [self.pt.append(r) for r in rids]
        if self.raw is not None:
            seen = []
            for r in rids:
                if r not in seen:
                    seen.append(r)
            self.raw.allocate_paged([(r, before[r], self.pt.length[r]) for r in seen])
        for x in res:
            if x["cow"] is not None:
                for layer in self.layers:
                    self.stores[layer].copy_page(x["cow"][0], x["cow"][1], self.sc.w.P)
        return [x["slot"] for x in res]

    def table_row(self, rid):
        """The device-visible prefix of a request's table row."""
        if self.raw is not None:
            n = len(self.pt.block_row(rid)) * self.sc.w.P
            return [int(x) for x in self.raw.page_table[rid, :n]]
        return self.pt.block_row(rid)

    def _op(self, op):
        kind = op[0]
        if kind == "new":
            self.pt.new(op[1])
        elif kind == "append":
            _, rid, n, store_from, store_below = op
            L0 = self.pt.length[rid]
            slots = self._append([rid] * n)
            first = max(store_from, L0)
            self._store(rid, list(range(first, L0 + n)), slots[first - L0:])
            sink_end = min(store_below, first, L0 + n)
            if L0 < sink_end:
                self._store(rid, list(range(L0, sink_end)), slots[:sink_end - L0])
        elif kind == "batch":
            pos = [self.pt.length[r] for r in op[1]]
            slots = self._append(op[1])
            for r, p, s in zip(op[1], pos, slots):
                self._store(r, [p], [s])
        elif kind == "trim":
            if op[3]:
                self.pt.trim(op[1], op[2], sink_rows=op[3])
            else:
                self.pt.trim(op[1], op[2])
        elif kind == "fork":
            self.pt.fork(op[1], op[2])
        elif kind == "release":
            self.pt.release(op[1])

    def _verify_step(self, step_index, attend_rids, with_slots, queries=None):
        """A speculative step: M drafts appended per request, the ones of
        ``attend_rids`` stored and verified, the seeded acceptance applied by
        rewinding the rest. ``queries``: the query indices j to attend (all
        when None; a timed sample of a long chunk takes a subset)."""
        sc, w, OA, M = self.sc, self.sc.w, self.OA, self.sc.multi
        pos0 = {r: self.pt.length[r] for r in sc.rids}
        rr = [r for r in sc.rids for _ in range(M)]
        slots = self._append(rr)
        outs = {}
        for r in attend_rids:
            i = sc.rids.index(r)
            self._store(r, [pos0[r] + j for j in range(M)], slots[i * M:(i + 1) * M])
        for r in attend_rids:
            L = self.pt.length[r]
            row = self.pt.block_row(r)
            for layer in self.layers:
                per_q = []
                for j, pos in enumerate(OA.verify_positions(L, M, sc.window, sc.sinks)):
                    if queries is not None and j not in queries:
                        continue
                    q = sc.inputs.q_rows(sc.seed, step_index * M + j, layer, [r], w.Hq, w.D, dtype=self.tdt)[0]
                    sl = [s for p in pos for s in OA.gather_block(row, w.P, p, p + 1)]
                    per_q.append(OA.attend_request(self.stores[layer], q.float().numpy(), sl, w.scale))
                outs[(r, layer)] = np.stack(per_q)
        if sc.verify:
            for r, a in zip(sc.rids, wl.accepted_drafts(sc.seed, step_index, len(sc.rids), M)):
                self.pt.rewind(r, M - a)
        return (outs, slots) if with_slots else outs

    def step(self, step_index, attend_rids, with_slots=False, queries=None):
        """One decode step: bookkeeping for every request, store + attention for ``attend_rids``.

        Returns {(rid, layer): output}, and also the step's slots when ``with_slots``."""
        if self.sc.multi:
            return self._verify_step(step_index, attend_rids, with_slots, queries)
        sc, w, OA = self.sc, self.sc.w, self.OA
        pos = [self.pt.length[r] for r in sc.rids]
        slots = self._append(sc.rids)
        by_rid = dict(zip(sc.rids, zip(pos, slots)))
        outs = {}
        for r in attend_rids:
            p, s = by_rid[r]
            self._store(r, [p], [s])
        for r in attend_rids:
            L = self.pt.length[r]
            pos = OA.attended_positions(L, sc.window, sc.sinks)
            for layer in self.layers:
                q = sc.inputs.q_rows(sc.seed, step_index, layer, [r], w.Hq, w.D, dtype=self.tdt)[0].float().numpy()
                if self.raw is not None:
                    row = self.raw.page_table[r]
                    sl = [s for p in pos for s in OA.gather_raw(row, p, p + 1)]
                else:
                    row = self.pt.block_row(r)
                    sl = [s for p in pos for s in OA.gather_block(row, w.P, p, p + 1)]
                outs[(r, layer)] = OA.attend_request(self.stores[layer], q, sl, w.scale)
        if sc.window > 0:
            for r in sc.rids:
                kf = max(0, self.pt.length[r] + 1 - (sc.window - sc.sinks))
                if sc.sinks:
                    self.pt.trim(r, kf, sink_rows=sc.sinks)
                else:
                    self.pt.trim(r, kf)
        return (outs, slots) if with_slots else outs


def _sample_rids(sc, n):
    # spread the sample over the batch (first, last and evenly between)
    B = len(sc.rids)
    idx = sorted({int(round(i * (B - 1) / max(1, n - 1))) for i in range(n)})
    return [sc.rids[i] for i in idx]


def timed_queries(sc):
    """Query tokens a timed oracle sample attends per request: all of a decode
    or verify step; 16 evenly spaced ones of a long prefill chunk, whose bytes
    are then credited in proportion. Returns (indices or None, fraction)."""
    M = max(sc.multi, 1)
    if M <= 32:
        return None, 1.0
    js = sorted({round(k * (M - 1) / 15) for k in range(16)})
    return set(js), len(js) / M


def cpu_baseline(sc, seconds):
    """The oracle, as it stands, on one host core: decode steps of a sample of
    requests of the same workload, timed for about ``seconds``."""
    n = 4 if sc.w.layers == 1 else 2
    sample = _sample_rids(sc, n)
    orc = OracleSample(sc, sample)
    queries, frac = timed_queries(sc)
    done_bytes, t_total, steps = 0, 0.0, 0
    while t_total < seconds or steps == 0:
        steps += 1
        t = time.perf_counter()
        orc.step(10_000 + steps, sample, queries=queries)
        t_total += time.perf_counter() - t
        lens = [orc.pt.length[r] for r in sample]
        done_bytes += frac * sc.w.layers * attention_bytes(sc, lens)
    return {
        "value": round(done_bytes / t_total / 1e9, 6),
        "unit": UNIT,
        "cores": 1,
        "kind": "oracle",
        "sample": f"{steps} decode steps of {len(sample)} of {len(sc.rids)} requests (all {sc.w.layers} layers); "
                  f"bookkeeping for every request, store + float64 attention for the sample"
                  + (f" ({len(queries)} of {sc.multi} query tokens each, bytes credited in proportion)"
                     if queries else ""),
        "seconds": round(t_total, 2),
    }


def _oracle_worker(name, seed, n_layers, layers, sample, seconds, barrier, out_q):
    """One process of the all-cores oracle timing: builds the workload's
    oracle state for its layers, waits for the others, then times decode
    steps of its own sample of requests for about ``seconds``."""
    try:
        sc = Scenario(name, seed, layers=n_layers)
        orc = OracleSample(sc, sample, layers=layers)
        queries, frac = timed_queries(sc)
        barrier.wait(timeout=600)
        done, t_total, steps = 0.0, 0.0, 0
        while t_total < seconds or steps == 0:
            steps += 1
            t = time.perf_counter()
            orc.step(10_000 + steps, sample, queries=queries)
            t_total += time.perf_counter() - t
            done += frac * len(orc.layers) * attention_bytes(sc, [orc.pt.length[r] for r in sample])
        out_q.put((done, t_total, steps, len(sample)))
    except Exception as e:  # reported to the parent, which then keeps the single-core figure
        out_q.put(repr(e))


def cpu_baseline_all_cores(sc, seconds, workers):
    """The oracle on ``workers`` host cores at once: one spawned process per
    core, timed together; the value is the sum of their rates. One-layer
    workloads give each process its own sample of requests (disjoint, spread
    over the batch); multi-layer workloads give each its own layers (the
    same two requests, every layer taken by one process), whose oracle state
    stays small."""
    import multiprocessing as mp

    ctx = mp.get_context("spawn")  # safe after CUDA has been initialised
    B, NL = len(sc.rids), sc.w.layers
    if NL == 1:
        per = max(1, min(4, B // workers))
        jobs = [([0], s) for s in ([sc.rids[i] for i in range(w, B, workers)][:per] for w in range(workers)) if s]
    else:
        per = 2
        sample = _sample_rids(sc, per)
        jobs = [(list(range(w, NL, workers)), sample) for w in range(min(workers, NL))]
    barrier, out_q = ctx.Barrier(len(jobs)), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(sc.name, sc.seed, NL, lay, smp, seconds, barrier, out_q),
                         daemon=True) for lay, smp in jobs]
    import queue

    for p in procs:
        p.start()
    res = []
    try:
        deadline = time.time() + 1200
        while len(res) < len(procs):
            try:
                res.append(out_q.get(timeout=1.0))
            except queue.Empty:
                # a process that died without reporting would leave the others at the barrier
                if any(p.exitcode not in (None, 0) for p in procs) or time.time() > deadline:
                    raise RuntimeError("an oracle process ended without a result")
    finally:
        for p in procs:
            p.join(timeout=5)
            if p.is_alive():
                p.kill()
    bad = [r for r in res if isinstance(r, str)]
    if bad:
        raise RuntimeError(bad[0])
    rate = sum(d / t for d, t, _, _ in res)
    steps = min(r[2] for r in res)
    return {
        "value": round(rate / 1e9, 6),
        "cores": len(procs),
        "sample": (f"{len(procs)} processes, each {steps}+ decode steps of its own {per} of {B} requests, timed "
                   f"together; rates summed" if NL == 1 else
                   f"{len(procs)} processes, each {steps}+ decode steps of the same {per} of {B} requests on its own "
                   f"{len(jobs[0][0])} of {NL} layers (every layer taken once), timed together; rates summed"),
    }


def run_reference(args):
    """--impl reference: the CPU oracle on the same workload, metric and unit."""
    sc = Scenario(args.workload, args.seed, layers=args.layers)
    n = 2 if sc.w.layers == 1 else 1
    sample = _sample_rids(sc, n)
    orc = OracleSample(sc, sample)
    queries, frac = timed_queries(sc)
    for i in range(args.warmup):
        orc.step(1 + i, sample, queries=queries)
    t = time.perf_counter()
    done = 0
    for i in range(args.steps):
        orc.step(1 + args.warmup + i, sample, queries=queries)
        done += frac * sc.w.layers * attention_bytes(sc, [orc.pt.length[r] for r in sample])
    el = time.perf_counter() - t
    value = done / el / 1e9
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": UNIT,
        "n_gpus": 0,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded workload as the GPU arm)",
        "config": {"workload": sc.name, "batch": len(sc.rids), "sampled_requests": len(sample),
                   "layers": sc.w.layers, "seed": args.seed},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{len(sample)} of {len(sc.rids)} requests per step, all layers"
                                   + (f", {len(queries)} of {sc.multi} query tokens each (bytes credited in "
                                      f"proportion)" if queries else "")},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed attention before warm-up")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the extra legs of the headline workload")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer count of the 32-layer workloads (a small variant for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    line = run_gpu(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
