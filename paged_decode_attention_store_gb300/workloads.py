"""Seeded synthetic inputs for the paged decode-attention workloads.

This module is the ONLY code that both the CUDA path (tests, bench) and the
CPU oracle consume. It holds none of the method's arithmetic: it produces
random values, lengths and permutations, nothing else.

Values
------
Every Q/K/V element is a pure function of ``(seed, stream, element index)``
(a counter-based generator), so any subset of rows can be produced on any
device, in any order, bit-identically. The recipe:

1. ``h = mix32(lo ^ mix32((hi + key) mod 2^32))`` where ``lo``/``hi`` are the
   low/high 32 bits of the element index, ``key`` mixes seed and stream, and
   ``mix32`` is the "lowbias32" integer hash published by C. Wellons (hash
   prospector): ``x ^= x>>16; x *= 0x7feb352d; x ^= x>>15; x *= 0x846ca68b;
   x ^= x>>16`` (mod 2^32).
2. The top 16 bits ``i = h >> 16`` pick one of 2^16 equiprobable levels of
   N(0, 1) by inverse transform sampling: the value is the standard normal
   quantile at the level's midpoint, ``Phi^-1((i + 0.5) / 2^16)``, from a
   table computed once in float64 (``statistics.NormalDist().inv_cdf``) and
   rounded to float32. The result is N(0, 1) up to a discretisation far
   below bf16 resolution; its support is +-4.33 (the standard normal puts
   1.5e-5 of its mass beyond that).
3. bf16 workloads round that float32 value to bf16 (round to nearest even).

All integer steps run in int64 tensors holding 32-bit values, with the
32-bit products split in 16-bit halves so that no step overflows, and the
quantile step is a table gather; torch gives the same bits on CPU and CUDA.

Element indices
---------------
``K/V``: ``((((layer*2 + kv)*2^12 + request)*2^20 + position)*2^6 + head)*2^9 + d``
``Q``:   ``((((step*2^6 + layer)*2^12 + request)*2^6 + head)*2^9 + d``

Lengths and permutations come from ``numpy.random.RandomState`` (whose
stream numpy keeps frozen across versions).
"""

from __future__ import annotations

import math
import statistics
from dataclasses import dataclass, field

import numpy as np
import torch

_M32 = 0xFFFFFFFF
STREAM_K, STREAM_V, STREAM_Q = 1, 2, 3


def _mul32_t(x: torch.Tensor, c: int) -> torch.Tensor:
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _mix32_t(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32_t(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32_t(x, 0x846CA68B)
    return x ^ (x >> 16)


def _mix32_i(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    return x ^ (x >> 16)


_LEVELS = 1 << 16
_QUANTILES = {}


def _quantile_table(device) -> torch.Tensor:
    """Standard normal quantiles at the midpoints of 2^16 equiprobable
    levels, float32, cached per device (built on the host, then copied)."""
    key = str(torch.device(device))
    t = _QUANTILES.get(key)
    if t is None:
        if "cpu" not in _QUANTILES:
            nd = statistics.NormalDist()
            _QUANTILES["cpu"] = torch.tensor([nd.inv_cdf((i + 0.5) / _LEVELS) for i in range(_LEVELS)],
                                             dtype=torch.float64).to(torch.float32)
        t = _QUANTILES["cpu"].to(device)
        _QUANTILES[key] = t
    return t


def hash_normal(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """float32 N(0,1) value (2^16-level inverse transform) for each int64 element index."""
    key = _mix32_i(_mix32_i(seed * 0x9E3779B9 + 0x632BE5AB) ^ (stream * 0x85EBCA77))
    lo = idx & _M32
    hi = idx >> 32
    h = _mix32_t(lo ^ _mix32_t((hi + key) & _M32))
    return _quantile_table(idx.device)[h >> 16]


def _as_index(x, device) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.int64, device=device).reshape(-1)


def kv_rows(seed: int, layer: int, rid, pos, Hkv: int, D: int,
            dtype=torch.bfloat16, device="cpu"):
    """K and V rows ``[n, Hkv, D]`` of tokens ``(rid[i], pos[i])`` in ``layer``.

    ``rid`` and ``pos`` are equal-length integer sequences (or one of them a
    scalar). Values depend only on (seed, layer, request, position, head, d).
    """
    rid = _as_index(rid, device)
    pos = _as_index(pos, device)
    rid, pos = torch.broadcast_tensors(rid, pos)
    assert Hkv <= 64 and D <= 512 and layer < 64
    h = torch.arange(Hkv, dtype=torch.int64, device=device).view(1, Hkv, 1)
    d = torch.arange(D, dtype=torch.int64, device=device).view(1, 1, D)
    out = []
    for kv, stream in ((0, STREAM_K), (1, STREAM_V)):
        base = ((layer * 2 + kv) * 4096 + rid) * (1 << 20) + pos
        idx = ((base.view(-1, 1, 1) * 64 + h) * 512) + d
        out.append(hash_normal(seed, stream, idx).to(dtype))
    return out[0], out[1]


def q_rows(seed: int, step: int, layer: int, rid, Hq: int, D: int,
           dtype=torch.bfloat16, device="cpu"):
    """Query rows ``[n, Hq, D]`` of requests ``rid`` at decode step ``step``."""
    rid = _as_index(rid, device)
    assert Hq <= 64 and D <= 512 and layer < 64
    h = torch.arange(Hq, dtype=torch.int64, device=device).view(1, Hq, 1)
    d = torch.arange(D, dtype=torch.int64, device=device).view(1, 1, D)
    base = (step * 64 + layer) * 4096 + rid
    idx = ((base.view(-1, 1, 1) * 64 + h) * 512) + d
    return hash_normal(seed, STREAM_Q, idx).to(dtype)


def permutation(seed: int, n: int) -> np.ndarray:
    return np.random.RandomState(seed).permutation(n).astype(np.int64)


def free_stack_for_order(order) -> list:
    """Free-list stack (top = end) that hands pages out in ``order``."""
    return [int(p) for p in reversed(list(order))]


# ---------------------------------------------------------------------------
# The five workloads. Each is a plain description: shapes, lengths and the
# initial free-list order; building tables from them is the method's job.
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16"
    Hq: int
    Hkv: int
    D: int
    P: int
    layers: int
    num_pages: int             # managed pages (the pool may add a dummy page)
    free_order: list           # free-list stack, top = end
    lengths: list              # context length of each request before the first decode step
    window: int = 0            # <= 0: none
    sinks: int = 0             # attention-sink rows kept in every windowed context
    scale: float = 0.0
    table_mode: str = "block"  # "block" or "raw"
    extra: dict = field(default_factory=dict)


def tiny(seed: int = 0, window=None) -> Workload:
    """1 layer, fp32, 2 q / 2 kv heads, head_dim 16, page 4, 64 pages; 4 requests
    decode 32 tokens each from empty; windows none / 8 / 4."""
    n_pages = 64
    return Workload("tiny", "f32", 2, 2, 16, 4, 1, n_pages,
                    free_stack_for_order(permutation(seed * 7919 + 11, n_pages)),
                    [0, 0, 0, 0], window=0 if window is None else window,
                    scale=1.0 / math.sqrt(16), extra={"steps": 32})


def gqa_decode(seed: int = 0) -> Workload:
    """bf16, 32 q / 8 kv heads, head_dim 128, page 16, batch 64, context
    lengths uniform in [512, 4096], pool = pages needed + 10%, block tables a
    seeded random permutation of the pages, no window."""
    P, B = 16, 64
    rs = np.random.RandomState(seed * 7919 + 2)
    lengths = rs.randint(512, 4096 + 1, size=B).tolist()
    need = sum(-(-L // P) for L in lengths)
    n_pages = int(math.ceil(need * 1.1))
    order = np.random.RandomState(seed * 7919 + 3).permutation(n_pages)
    return Workload("gqa_decode", "bf16", 32, 8, 128, P, 1, n_pages,
                    free_stack_for_order(order), lengths, scale=1.0 / math.sqrt(128))


def gqa_verify(seed: int = 0, M: int = 4) -> Workload:
    """gqa_decode's requests in speculative decoding: every step appends M
    drafted tokens per request, verifies them at once, accepts a seeded
    uniform number in [0, M] and rewinds the rest. The pool adds 16 pages
    per request for the growth over a run."""
    w = gqa_decode(seed)
    n_pages = w.num_pages + 16 * len(w.lengths)
    order = np.random.RandomState(seed * 7919 + 3).permutation(n_pages)
    return Workload(f"gqa_verify{M}", "bf16", w.Hq, w.Hkv, w.D, w.P, 1, n_pages, free_stack_for_order(order),
                    list(w.lengths), scale=w.scale, extra={"verify": M})


def gqa_prefill(seed: int = 0, chunk: int = 512) -> Workload:
    """Chunked prefill with gqa_decode's heads: bf16, 32 q / 8 kv heads,
    head_dim 128, page 16, 16 requests with a prefix uniform in [0, 2048];
    every step appends a chunk of ``chunk`` tokens per request, stores it and
    attends it at once (causal). The pool holds 72 chunks of growth."""
    P, B = 16, 16
    rs = np.random.RandomState(seed * 7919 + 12)
    lengths = rs.randint(0, 2048 + 1, size=B).tolist()
    n_pages = sum(-(-(L + 72 * chunk) // P) for L in lengths) + B
    order = np.random.RandomState(seed * 7919 + 13).permutation(n_pages)
    return Workload(f"gqa_prefill{chunk}", "bf16", 32, 8, 128, P, 1, n_pages, free_stack_for_order(order), lengths,
                    scale=1.0 / math.sqrt(128), extra={"prefill": chunk})


def accepted_drafts(seed: int, step: int, B: int, M: int) -> list:
    """Drafts accepted per request at a verify step: uniform in [0, M]."""
    return np.random.RandomState(seed * 7919 + 1000 + step).randint(0, M + 1, size=B).tolist()


def sliding_window(seed: int = 0) -> Workload:
    """bf16, 32 q / 8 kv heads, head_dim 128, page 16, batch 32, W = 4096,
    context lengths uniform in [8192, 32768]; pages older than the window are
    released (front holes), at most ceil((W-1)/16)+1 live pages per request."""
    P, B, W = 16, 32, 4096
    rs = np.random.RandomState(seed * 7919 + 4)
    lengths = rs.randint(8192, 32768 + 1, size=B).tolist()
    live = -(-(W - 1) // P) + 1
    n_pages = int(math.ceil(B * live * 1.1))
    order = np.random.RandomState(seed * 7919 + 5).permutation(n_pages)
    return Workload("sliding_window", "bf16", 32, 8, 128, P, 1, n_pages,
                    free_stack_for_order(order), lengths, window=W,
                    scale=1.0 / math.sqrt(128))


def sliding_window_sinks(seed: int = 0, sinks: int = 2) -> Workload:
    """sliding_window with attention sinks (chapter 15, exercise "Attention
    sinks": the first 2 rows plus the last W - 2): the same lengths and pool,
    the first page of each request kept past the window."""
    w = sliding_window(seed)
    P, B = w.P, len(w.lengths)
    live = -(-sinks // P) + -(-(w.window - sinks - 1) // P) + 1
    n_pages = int(math.ceil(B * live * 1.1))
    order = np.random.RandomState(seed * 7919 + 5).permutation(n_pages)
    return Workload("sliding_window_sinks", "bf16", w.Hq, w.Hkv, w.D, P, 1, n_pages,
                    free_stack_for_order(order), list(w.lengths), window=w.window, sinks=sinks,
                    scale=w.scale)


def prefix_sharing(seed: int = 0) -> Workload:
    """bf16, 32 q / 8 kv heads, head_dim 128, page 16: 8 prompts of 2050 tokens,
    each forked 16 times (128 requests); private suffixes uniform in [16, 512]."""
    P, n_prompts, forks, prompt_len = 16, 8, 16, 2050
    rs = np.random.RandomState(seed * 7919 + 6)
    suffix = rs.randint(16, 512 + 1, size=n_prompts * forks).tolist()
    shared = n_prompts * -(-prompt_len // P)
    private = sum(-(-(prompt_len + s + 256) // P) - prompt_len // P for s in suffix)
    n_pages = int(math.ceil((shared + private) * 1.1))
    order = np.random.RandomState(seed * 7919 + 7).permutation(n_pages)
    lengths = [prompt_len + s for s in suffix]
    return Workload("prefix_sharing", "bf16", 32, 8, 128, P, 1, n_pages,
                    free_stack_for_order(order), lengths, scale=1.0 / math.sqrt(128),
                    extra={"n_prompts": n_prompts, "forks": forks,
                           "prompt_len": prompt_len, "suffix": suffix})


def large_batch(seed: int = 0, P: int = 16, headroom: int = 256, layers: int = 32, lengths=None) -> Workload:
    """mini-sglang layout: bf16, 64 q / 8 kv heads, head_dim 128, batch 256,
    32 layers, context lengths lognormal (median 1024, sigma 0.8) capped at
    16384 (minus ``headroom`` decode steps), raw token-location page table of
    shape (257, align32(16384)), run at page 16 and page 1. ``layers`` and
    ``lengths`` (a replacement list of 256 lengths) make variants of it."""
    B, max_seq = 256, 16384
    rs = np.random.RandomState(seed * 7919 + 8)
    draw = rs.lognormal(mean=math.log(1024.0), sigma=0.8, size=B)
    if lengths is None:
        lengths = [int(min(max_seq - headroom, max(1, math.floor(x + 0.5)))) for x in draw]
    lengths = [int(L) for L in lengths]
    assert len(lengths) == B and all(1 <= L <= max_seq - headroom for L in lengths)
    need = sum(-(-(L + headroom) // P) for L in lengths)
    n_pages = int(math.ceil(need * 1.1))
    order = np.random.RandomState(seed * 7919 + 9 + P).permutation(n_pages)
    return Workload(f"large_batch_p{P}", "bf16", 64, 8, 128, P, layers, n_pages,
                    free_stack_for_order(order), lengths, scale=1.0 / math.sqrt(128),
                    table_mode="raw",
                    extra={"max_running_req": B, "max_seq_len": max_seq,
                           "headroom": headroom})


class CodedInputs:
    """Structured inputs whose attention outputs show which K/V rows were read.

    K and the odd query heads come from the seeded generator above; the even
    query heads are zero, so their scores are all equal. Each V row holds
    two ones and zeros elsewhere, placed by the token's position ``t`` over
    the ``Hkv * D`` entries of a row (``half = D / 2`` entries per head):

    - row code: entry ``(h, d)`` with ``h * half + d = t mod (Hkv * half)``;
    - stage code: entry ``(h, half + d)`` with ``h * half + d = (t div 16)
      mod (Hkv * half)``, one entry per 16-position group.

    The values are exact in bf16. Every output entry is then a weighted count
    of the attended rows of one residue class, so a row or a 16-row group that
    is read twice, skipped or taken from another position moves an entry by a
    whole row's weight.
    """

    STAGE = 16

    def kv_rows(self, seed, layer, rid, pos, Hkv, D, dtype=torch.bfloat16, device="cpu"):
        k, _ = kv_rows(seed, layer, rid, pos, Hkv, D, dtype=dtype, device=device)
        rid = _as_index(rid, device)
        pos = _as_index(pos, device)
        rid, pos = torch.broadcast_tensors(rid, pos)
        half = D // 2
        n = pos.numel()
        v = torch.zeros((n, Hkv * D), dtype=dtype, device=device)
        rows = torch.arange(n, device=device)
        c = pos % (Hkv * half)
        v[rows, (c // half) * D + c % half] = 1
        c = (pos // self.STAGE) % (Hkv * half)
        v[rows, (c // half) * D + half + c % half] = 1
        return k, v.view(n, Hkv, D)

    def q_rows(self, seed, step, layer, rid, Hq, D, dtype=torch.bfloat16, device="cpu"):
        q = q_rows(seed, step, layer, rid, Hq, D, dtype=dtype, device=device)
        q[:, 0::2, :] = 0
        return q
