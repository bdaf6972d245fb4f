"""The prefill trace report's arithmetic, on synthetic records (no GPU).

CTAs on 4 SMs last exactly 3 us + 1 us per key block with 0.5 us between
consecutive CTAs of an SM; the armed CTA's events follow a fixed pattern per
block. The fit, the gaps and the steady-state medians must come back as
built."""

import numpy as np

from paged_decode_attention_store_gb300 import trace_prefill as tp


def _records():
    ctas = np.zeros((4096, 4), np.uint64)
    t_sm = [1_000_000] * 4
    nblocks = [5, 9, 12, 7, 20, 3, 11, 6]
    for c, nb in enumerate(nblocks):
        sm = c % 4
        start = t_sm[sm]
        end = start + 3000 + 1000 * nb
        ctas[c] = (start, sm, end, nb)
        t_sm[sm] = end + 500
    ev = np.zeros((len(tp.EVENTS), 128), np.uint64)
    cta = 4  # 20 blocks
    b0 = int(ctas[cta, 0])
    offsets = {"k_resolved": 100, "k_issued": 300, "v_resolved": 150, "v_issued": 350, "s_kfull": 500,
               "s_issued": 700, "pv_vfull": 800, "sm_sfull": 900, "sm_max": 1100, "sm_p": 1400, "sm_arrive": 1500,
               "pv_pfull": 1600, "pv_issued": 1900}
    for i in range(int(ctas[cta, 3])):
        for name, off in offsets.items():
            ev[tp.E[name], i] = b0 + 2000 + 1000 * i + off
    return ev, ctas, cta


def test_trace_report_recovers_the_built_timings():
    ev, ctas, cta = _records()
    lines = tp.analyse(ev, ctas, 4, cta)
    text = "\n".join(lines)
    assert "3.00 us fixed + 1.000 us per key block" in text, text
    assert "gap between CTAs on an SM: median 0.50 us" in text, text
    assert "s_kfull->s_issued 0.20" in text and "sm_max->sm_p 0.30" in text and "pv_pfull->pv_issued 0.30" in text
    assert "k_resolved->k_issued 0.20" in text and "v_issued->pv_vfull 0.45" in text
    assert "block period (softmax sees S(i) to S(i + 1)): median 1.00 us" in text, text


def test_trace_report_refuses_a_short_cta():
    ev, ctas, _ = _records()
    lines = tp.analyse(ev, ctas, 4, 5)  # 3 blocks
    assert "too few for a steady state" in lines[-1]
