"""Per-stage timing of the chunked-prefill kernel's pipeline on the GPU.

Builds the tracing variant of the library (prefill_tc.cu compiled with
KVP_PREFILL_TRACE: every CTA records its entry and exit times, SM and key
blocks, and one armed CTA the global-timer time of each pipeline event of
its key blocks), runs the first steps of the ``gqa_prefill512`` workload
through the bench's scenario on cuda:0, arms one CTA for the last of them
and prints:

- every CTA's duration fitted as a fixed cost plus a cost per key block,
  the gap between consecutive CTAs on an SM, the launch's tail and how busy
  the SMs were;
- for the armed CTA, the first events after its entry, the time from its
  last P V issue to its exit, and the median time between pipeline events
  over its steady-state blocks (2 .. n - 1), with the block period.

    python -m paged_decode_attention_store_gb300.trace_prefill [--steps N] [--cta C]

The product library is never the traced one; this is a measuring tool.
"""

from __future__ import annotations

import argparse
import ctypes
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# the kernel's event order (enum PrefillTraceEvent in prefill_tc.cu)
EVENTS = ["k_resolved", "k_issued", "v_resolved", "v_issued", "s_kfull", "s_issued", "pv_vfull", "pv_pfull",
          "pv_issued", "sm_sfull", "sm_max", "sm_p", "sm_arrive"]
E = {name: i for i, name in enumerate(EVENTS)}

# consecutive pipeline events of one block whose median gaps are printed
CHAIN = [("s_kfull", "s_issued"), ("s_issued", "sm_sfull"), ("sm_sfull", "sm_max"), ("sm_max", "sm_p"),
         ("sm_p", "sm_arrive"), ("sm_arrive", "pv_pfull"), ("pv_pfull", "pv_issued")]
LOADS = [("k_resolved", "k_issued"), ("k_issued", "s_kfull"), ("v_resolved", "v_issued"), ("v_issued", "pv_vfull")]


def _trace_lib():
    from . import binding as kb
    from . import build as kbuild

    kb.LIB_PATH = kbuild.build_traced()
    lib = kb.lib()
    lib.kvp_prefill_trace_arm.argtypes = [ctypes.c_int]
    lib.kvp_prefill_trace_arm.restype = ctypes.c_int
    lib.kvp_prefill_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.kvp_prefill_trace_read.restype = ctypes.c_int
    return lib


def analyse(ev, ctas, n_sms, cta):
    """The printed report from the raw records (times in ns)."""
    import numpy as np

    lines = []
    live = ctas[:, 3] > 0
    c = ctas[live].astype(np.int64)
    t0 = c[:, 0].min()
    dur = (c[:, 2] - c[:, 0]) / 1e3
    nb = c[:, 3].astype(float)
    span = (c[:, 2].max() - t0) / 1e3
    coef, *_ = np.linalg.lstsq(np.stack([np.ones_like(nb), nb], 1), dur, rcond=None)
    gaps = []
    for sm in np.unique(c[:, 1]):
        rows = c[c[:, 1] == sm]
        rows = rows[np.argsort(rows[:, 0])]
        gaps += list((rows[1:, 0] - rows[:-1, 2]) / 1e3)
    last_end = [c[c[:, 1] == sm, 2].max() for sm in np.unique(c[:, 1])]
    lines.append(f"launch: {len(c)} CTAs over {span:.1f} us; SMs busy {dur.sum() / (n_sms * span):.3f} of the span; "
                 f"tail (last SM done - first SM done) {(max(last_end) - min(last_end)) / 1e3:.1f} us")
    lines.append(f"CTA duration: {coef[0]:.2f} us fixed + {coef[1]:.3f} us per key block "
                 f"(blocks {int(nb.min())}..{int(nb.max())}, median {np.median(nb):.0f}); "
                 f"gap between CTAs on an SM: median {np.median(gaps):.2f} us")
    e = ev.astype(np.int64)
    b0 = ctas[cta, 0].astype(np.int64)
    n = int(min(ctas[cta, 3], e.shape[1]))
    if n < 4:
        lines.append(f"CTA {cta}: {n} key blocks, too few for a steady state")
        return lines
    rel = lambda name, i: (e[E[name], i] - b0) / 1e3  # noqa: E731
    lines.append(f"CTA {cta} ({n} key blocks, {(ctas[cta, 2] - ctas[cta, 0]) / 1e3:.1f} us): first K copies issued "
                 f"{rel('k_issued', 0):.2f} us after entry, first S {rel('s_issued', 0):.2f}, first softmax "
                 f"{rel('sm_sfull', 0):.2f}; last P V issued {(ctas[cta, 2] - e[E['pv_issued'], n - 1]) / 1e3:.2f} "
                 f"us before exit")

    def med(a, b):
        return float(np.median((e[E[b], 2:n] - e[E[a], 2:n]) / 1e3))

    lines.append("steady state, median us: " + " | ".join(f"{a}->{b} {med(a, b):.2f}" for a, b in CHAIN))
    lines.append("loads, median us: " + " | ".join(f"{a}->{b} {med(a, b):.2f}" for a, b in LOADS))
    lines.append(f"block period (softmax sees S(i) to S(i + 1)): median "
                 f"{float(np.median(np.diff(e[E['sm_sfull'], 2:n]) / 1e3)):.2f} us")
    return lines


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--steps", type=int, default=5, help="prefill steps; the last one is traced")
    ap.add_argument("--cta", type=int, default=None, help="CTA to arm (default: one of request 5)")
    args = ap.parse_args(argv)

    import numpy as np
    import torch

    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    lib = _trace_lib()
    import bench

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    sc = bench.Scenario("gqa_prefill512", 0)
    w = sc.w
    tiles_per_head = -(-w.extra["prefill"] // (128 // (w.Hq // w.Hkv)))
    cta = args.cta if args.cta is not None else tiles_per_head * w.Hkv * 5 + 1
    cache, lens = bench.build_product(sc, dev)
    steps, _ = bench.prepare_steps(sc, cache, lens, 1, args.steps, dev)
    outs = [torch.empty(bench.out_shape(sc), dtype=cache.tdt, device=dev) for _ in range(w.layers)]
    assert lib.kvp_prefill_trace_arm(-1) == 0
    for st in steps[:-1]:
        bench.run_step(sc, cache, st, outs)
    torch.cuda.synchronize(dev)
    assert lib.kvp_prefill_trace_arm(cta) == 0
    bench.run_step(sc, cache, steps[-1], outs)
    torch.cuda.synchronize(dev)
    dims = np.zeros(3, np.int32)
    ev = np.zeros((len(EVENTS), 128), np.uint64)
    ctas = np.zeros((4096, 4), np.uint64)
    assert lib.kvp_prefill_trace_read(ev.ctypes.data, ctas.ctypes.data, dims.ctypes.data) == 0
    assert tuple(dims) == (len(EVENTS), 128, 4096), f"trace layout {tuple(dims)}"
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    print(f"gqa_prefill512, step {args.steps} (contexts prefix + {args.steps} x {w.extra['prefill']}), "
          f"traced library {os.path.basename(bench_lib_path())}")
    for line in analyse(ev, ctas, n_sms, cta):
        print(line)


def bench_lib_path():
    from . import binding as kb

    return kb.LIB_PATH


if __name__ == "__main__":
    main()
