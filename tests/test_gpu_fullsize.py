"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (same scenario scripts, same per-step device calls).

Bit-exact for every request: the slots each decode step writes and the
device table rows. Attention: every layer checked (32-layer workloads:
three layers) for a sample of requests spread over the batch, each output
computed one by one by the oracle, max |gpu - oracle| <= 2e-2 (bf16).
"""

import gc

import pytest
import torch

import bench
from gpu_harness import close
from libbuild import ensure_built

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def kb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_built()


@pytest.mark.parametrize("workload", bench.WORKLOADS)
def test_full_size_parity(kb, workload):
    sc = bench.Scenario(workload, 0)
    n_sample = 3
    sample = bench._sample_rids(sc, n_sample)
    track = set(sample)
    if workload == "prefix_sharing":  # the shared prompts are stored under the prompt requests
        x = sc.w.extra
        track |= {len(sc.rids) + f // x["forks"] for f in sample}
    layers = list(range(sc.w.layers)) if sc.w.layers == 1 else [0, sc.w.layers // 2, sc.w.layers - 1]
    orc = bench.OracleSample(sc, track, layers=layers)
    cache, lens = bench.build_product(sc, dev=DEV)
    steps, _ = bench.prepare_steps(sc, cache, lens, 1, 2, DEV)
    outs = [torch.empty(bench.out_shape(sc), dtype=cache.tdt, device=DEV) for _ in range(sc.w.layers)]
    for i, st in enumerate(steps):
        bench.run_step(sc, cache, st, outs)
        torch.cuda.synchronize(DEV)
        ref, slots = orc.step(i + 1, sample, with_slots=True)
        if sc.devalloc:  # the slots were chosen on the device, inside the step
            got_slots = cache._scratch[len(sc.rids)][:len(sc.rids)].cpu().tolist()
        else:
            got_slots = st.out_loc.cpu().tolist()
        assert got_slots == slots, "decode-step slots differ"
        got = {layer: outs[layer].float().cpu().numpy() for layer in layers}
        for r in sample:
            b = sc.rids.index(r)
            for layer in layers:
                close(got[layer][b], ref[(r, layer)], "bf16", f"{workload} step {i + 1} request {r} layer {layer}")
    tab = cache.table.cpu().numpy()
    for r in sc.rids:
        row = orc.table_row(r)
        assert tab[r, :len(row)].tolist() == row, f"table row {r}"
    if sc.devalloc:  # the device free list and counts equal the oracle's
        free, ref, lens_d, _, _ = cache.pages.snapshot()
        assert free == orc.pt.free and ref == orc.pt.ref
        assert [lens_d[r] for r in sc.rids] == [orc.pt.length[r] for r in sc.rids]
    cache.check()
    del cache, steps, outs
    gc.collect()
    torch.cuda.empty_cache()
