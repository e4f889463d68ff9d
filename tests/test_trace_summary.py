"""The step-timeline summary (host arithmetic only, CPU): per phase kind, averaged over
the layers, from a hand-built trace whose answers are known."""
from __future__ import annotations

import numpy as np
import pytest

from memory_bound_decode_dequant_gb300.trace import summarise


def test_summary_of_a_hand_built_trace():
    n_layers, ctas = 2, 3
    phases = 5 * n_layers + 1
    t = np.zeros((phases, ctas, 5), np.int64)
    base = 10_000_000  # the summary measures from the earliest entry stamp
    clock = base
    for p in range(phases):
        for c in range(ctas):
            arrive = clock + 1000 * c          # inputs arrive 0, 1, 2 us apart
            t[p, c] = [clock, arrive, arrive + 500, arrive + 500 + 2000 * (c + 1), 0]
            t[p, c, 4] = t[p, c, 3] + 250
        clock = int(t[p, :, 4].max())
    s = summarise(t, n_layers)
    assert set(s) == {"qkv", "attn", "o", "gu", "down", "head", "step_us"}
    for kind in ("qkv", "attn", "o", "gu", "down", "head"):
        k = s[kind]
        assert k["input_spread"] == pytest.approx(2.0)
        assert k["staging"] == pytest.approx(0.5)
        assert k["stream_mean"] == pytest.approx(4.0)   # (2 + 4 + 6) / 3
        assert k["stream_max"] == pytest.approx(6.0)
        assert k["epilogue"] == pytest.approx(0.25)
        assert k["span"] == pytest.approx(2.0 + 0.5 + 6.0 + 0.25)
    assert s["step_us"] == pytest.approx((clock - base) / 1e3, abs=0.05)


def test_layers_are_averaged_per_kind():
    n_layers, ctas = 2, 1
    t = np.zeros((11, ctas, 5), np.int64)
    for p in range(11):
        stream = 1000 if p < 5 else 3000  # layer 0 streams 1 us, layer 1 3 us
        t[p, 0] = [0, 0, 0, stream, stream]
    s = summarise(t, n_layers)
    assert s["qkv"]["stream_mean"] == pytest.approx(2.0)
    assert s["head"]["stream_mean"] == pytest.approx(3.0)


def test_stage_summary_of_a_hand_built_trace():
    """Two phases' worth of stages on one CTA: the stages are assigned to the phase whose
    streaming window holds their wait start; lead, wait, stall fraction, latency and
    math come out as built."""
    from memory_bound_decode_dequant_gb300.trace import summarise_stages
    n_layers = 1
    t = np.zeros((6, 1, 5), np.int64)
    t[0, 0] = [0, 0, 10_000, 20_000, 20_000]      # qkv streams in [10, 20] us
    t[3, 0] = [0, 0, 30_000, 40_000, 40_000]      # gate/up streams in [30, 40] us
    st = np.zeros((1, 1024, 4), np.int64)
    # qkv: two stages issued 5 us early, landed before they were wanted (no stall)
    st[0, 0] = [5_000, 10_000, 10_050, 10_550]
    st[0, 1] = [6_000, 11_000, 11_050, 11_550]
    # gate/up: one stage waited 2 us (issued 1 us before the wait began), one did not
    st[0, 2] = [29_000, 30_000, 32_000, 32_500]
    st[0, 3] = [29_500, 33_000, 33_000, 33_500]
    s = summarise_stages(t, st, n_layers)
    assert set(s) == {"qkv", "gu"}
    assert s["qkv"]["n"] == 2 and s["gu"]["n"] == 2
    assert s["qkv"]["lead"] == pytest.approx(5.0)
    assert s["qkv"]["wait"] == pytest.approx(0.05)
    assert s["qkv"]["stalled"] == pytest.approx(0.0) and s["qkv"]["latency"] is None
    assert s["qkv"]["math"] == pytest.approx(0.5)
    assert s["gu"]["lead"] == pytest.approx((1.0 + 3.5) / 2)
    assert s["gu"]["wait"] == pytest.approx(1.0)
    assert s["gu"]["stalled"] == pytest.approx(0.5)
    assert s["gu"]["latency"] == pytest.approx(3.0)
