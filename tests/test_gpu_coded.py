"""Full-size parity with position-coded inputs: a lost, doubled or misplaced
row or 16-row stage shows.

With random inputs the decode outputs shrink like 1/sqrt(L), and at long
contexts a 16-row group read twice or skipped at a split boundary moves them
by less than the 2e-2 bound of the random-input tests. Here the V rows are
one-hot codes of the token's position (row code: position mod 512 over the
8 KV heads x 64 entries; stage code: position div 16, likewise) and half the
query heads are zero (``workloads.CodedInputs``). A zero query head gives
every attended row the same weight, so its output is the exact count of
attended rows in each residue class divided by the number attended: the
oracle's closed form for equal scores. The other heads weight the same
counts by softmax weights of random keys.

Each workload runs in the launch configuration bench.py times (its
scenario script, the same per-step calls), two steps, and EVERY request's
output is compared element by element with the oracle (dense attention over
the rows of its attended positions, ``oracle.attention``), with a bound
relative to each entry: |gpu - oracle| <= rel |oracle| + 2^-20. bf16 rounds
to within 2^-8 of a value (its unit roundoff). A zero query head's output is
an exact count over an exact count, rounded once: rel = 1.25 * 2^-8 there.
The other heads also carry the bf16 rounding of every softmax weight, in
numerator and denominator alike: rel = 4 * 2^-8. A missing or extra row
moves an entry of a zero query head by at least 1/33 of it (7.8 * 2^-8) at
16,128 rows, a stage by far more.

The 32-layer workloads run one layer (the per-layer kernels are the same)
with three requests moved to the longest contexts the table admits
(16,128 rows, 16,127 and 8,193).
"""

import gc
import os

import numpy as np
import pytest
import torch

import bench
import oracle.attention as OA
from gpu_harness import RATIOS
from libbuild import ensure_built
from paged_decode_attention_store_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
REL_ZERO_Q, REL_RANDOM_Q, ABS = 1.25 * 2.0 ** -8, 4.0 * 2.0 ** -8, 2.0 ** -20
WORKLOADS = ["gqa_decode", "sliding_window", "sliding_window_sinks", "prefix_sharing", "large_batch_p16",
             "large_batch_p1", "gqa_verify4", "gqa_prefill512", "gqa_decode_devalloc"]


@pytest.fixture(scope="module")
def kb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_built()


def _scenario(name):
    inputs = wl.CodedInputs()
    if name.startswith("large_batch_p"):
        lens = list(wl.large_batch(0, P=int(name[len("large_batch_p"):])).lengths)
        lens[:3] = [16128, 16127, 8193]
        return bench.Scenario(name, 0, layers=1, inputs=inputs, lengths=lens)
    return bench.Scenario(name, 0, inputs=inputs)


def _source(sc, rid, positions):
    """(rid, position) keys whose generated rows sit at ``positions`` of
    request ``rid``: forks of a shared prompt read the prompt's rows below
    the prompt length (they were stored under the prompt request)."""
    if sc.name != "prefix_sharing":
        return [rid] * len(positions), list(positions)
    x = sc.w.extra
    owner = len(sc.rids) + rid // x["forks"]
    return [owner if t < x["prompt_len"] else rid for t in positions], list(positions)


class KRows:
    """K/V rows of the attended positions of each request (CPU, generated
    once per request and reused by the next step, which reads nearly the
    same positions)."""

    def __init__(self, sc):
        self.sc, self.rows = sc, {}

    def get(self, rid, pos, extra):
        pos = np.asarray(pos, np.int64)
        have = self.rows.get(rid)
        if have is None or not np.isin(pos, have[0]).all():
            w = self.sc.w
            want = np.union1d(pos, np.arange(pos.max() + 1, pos.max() + 1 + extra))
            r, p = _source(self.sc, rid, want.tolist())
            k, v = self.sc.inputs.kv_rows(self.sc.seed, 0, r, p, w.Hkv, w.D)
            have = self.rows[rid] = (want, k, v)
        idx = torch.from_numpy(np.searchsorted(have[0], pos))
        return have[1][idx].double().numpy(), have[2][idx].double().numpy()


def _expected(sc, krows, rid, L, step_index, queries):
    """Oracle outputs of request ``rid`` at a step with context ``L``:
    [Hq, D], or [M, Hq, D] for the given query indices of a multi-token step."""
    w, M = sc.w, max(sc.multi, 1)
    if not sc.multi:
        pos = OA.attended_positions(L, sc.window, sc.sinks)
        K, V = krows.get(rid, pos, 2)
        q = sc.inputs.q_rows(sc.seed, step_index, 0, [rid], w.Hq, w.D)[0].double().numpy()
        return OA.decode_attention(q, K, V, w.scale)
    outs = []
    for j, pos in enumerate(OA.verify_positions(L, M, sc.window, sc.sinks)):
        if j not in queries:
            continue
        K, V = krows.get(rid, pos, 2 * M)
        q = sc.inputs.q_rows(sc.seed, step_index * M + j, 0, [rid], w.Hq, w.D)[0].double().numpy()
        outs.append(OA.decode_attention(q, K, V, w.scale))
    return np.stack(outs)


def rel_bound(shape):
    """Per-entry relative bound of an output [..., Hq, D]: the even (zero)
    query heads REL_ZERO_Q, the odd ones REL_RANDOM_Q."""
    rel = np.full(shape, REL_RANDOM_Q)
    rel[..., 0::2, :] = REL_ZERO_Q
    return rel


def _check(got, ref, what):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    for name, heads in (("zero q", slice(0, None, 2)), ("random q", slice(1, None, 2))):
        e, r = err[..., heads, :], ref[..., heads, :]
        nz = r != 0
        if nz.any():  # the largest error relative to its entry, printed at the end of the run
            key = f"coded {name} rel err / 2^-8: " + os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
            RATIOS[key] = max(RATIOS.get(key, 0.0), float((e[nz] / np.abs(r[nz])).max()) / 2.0 ** -8)
    bad = err > rel_bound(ref.shape) * np.abs(ref) + ABS
    if bad.any():
        idx = tuple(int(i) for i in np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} entries off, first at {idx}: gpu {got[idx]!r} "
                             f"oracle {ref[idx]!r}")


@pytest.mark.parametrize("workload", WORKLOADS)
def test_coded_full_size_parity(kb, workload):
    sc = _scenario(workload)
    cache, lens = bench.build_product(sc, dev=DEV)
    steps, _ = bench.prepare_steps(sc, cache, lens, 1, 2, DEV)
    outs = [torch.empty(bench.out_shape(sc), dtype=cache.tdt, device=DEV) for _ in range(sc.w.layers)]
    krows = KRows(sc)
    # a prefill chunk: every query token of four requests spread over the
    # batch, and 16 query tokens of every other request
    M = max(sc.multi, 1)
    full = set(bench._sample_rids(sc, 4)) if sc.prefill else set(sc.rids)
    spread = set(round(i * (M - 1) / 15) for i in range(16)) if M > 16 else set(range(M))
    checked = 0
    for i, st in enumerate(steps):
        bench.run_step(sc, cache, st, outs)
        torch.cuda.synchronize(DEV)
        got = outs[0].float().cpu().numpy()
        for b, r in enumerate(sc.rids):
            queries = set(range(M)) if r in full else spread
            ref = _expected(sc, krows, r, st.lens_list[b], i + 1, queries)
            g = got[b] if not sc.multi else got[b][sorted(queries)]
            _check(g, ref, f"{workload} step {i + 1} request {r} (context {st.lens_list[b]})")
            checked += 1
    assert checked == 2 * len(sc.rids)
    cache.check()
    del cache, steps, outs
    gc.collect()
    torch.cuda.empty_cache()
