"""bench.py's FLOP accounting and needed K/V range against the oracle."""
import numpy as np
import pytest

import bench
import oracle
from sliding_window_attention_device_gb300 import synth


@pytest.mark.parametrize("layout,B,S,cp,window", [
    (("uniform", 5, 300, 50), 2, 2048, 4, 0),
    (("uniform", 5, 300, 50), 2, 2048, 8, 64),
    (("single",), 1, 1024, 4, 0),
    (("explicit", (100, 90, 50), 16), 1, 256, 4, 0),
    (("lognormal", 200.0, 1.0, 8, 900, 60), 3, 2048, 2, 300),
])
def test_pairs_and_needed_range_match_oracle(layout, B, S, cp, window):
    doc = synth.doc_layout(layout, B, S, 1)
    L = S // cp
    for r in range(cp):
        g = oracle.geom(B, 1, 1, 64, S, L, r * L, 0, S, window)
        assert bench.pairs_closed_form(doc, r * L, L, window) == oracle.pairs(doc, g)
        segs = oracle.segments(doc, g)
        real = [s for s in segs if s["n_real"] > 0]
        kvo, skv = bench.needed_range(doc, r * L, L)
        if real:
            assert kvo == min(s["s_first"] for s in real)
            assert kvo + skv == max(s["real_end"] for s in real)


def test_headline_pair_count_is_stable():
    w = synth.WORKLOADS["C2"]
    doc = synth.doc_layout(w.layout, w.B, w.S, 0)
    plan = bench.shard_plan(w, doc)
    assert len(plan) == 8
    total = sum(p["pairs"] for p in plan)
    g = oracle.geom(w.B, 1, 1, 128, w.S, w.L, 3 * w.L, 0, w.S)
    assert plan[3]["pairs"] == oracle.pairs(doc, g)
    assert total > 0


def test_peak_follows_the_clock_record():
    """Burst peak when the timed region ran at the maximum SM clock with no power
    cap; the sustained (power-capped) peak otherwise or when clocks are unknown."""
    peaks = {"source": "measured", "bf16_tflops": 1891.6, "bf16_tflops_sustained": 1686.5}
    p, src = bench.choose_peak(peaks, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert p == 1891.6 and "burst" in src
    assert round(792.8 / p, 2) == 0.42
    for clocks in ({"sm_mhz": 1432.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]},
                   {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]},
                   {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": []},
                   {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}):
        p, src = bench.choose_peak(peaks, clocks)
        assert p == 1686.5 and "sustained" in src, clocks


def test_end_to_end_bound():
    """The end-to-end bound is the slowest of the device step and the two copy
    directions at their measured rates (C2: 5.9 GB out at 193 GB/s)."""
    assert bench.e2e_bound_ms(9.75, 1.342e9, 5.914e9, 210.0, 193.0) == pytest.approx(30.64, abs=0.01)
    assert bench.e2e_bound_ms(50.0, 1e9, 1e9, 200.0, 200.0) == 50.0  # device-bound
    assert bench.e2e_bound_ms(1.0, 4e9, 1e9, 200.0, 200.0) == pytest.approx(20.0)  # host-to-device-bound
