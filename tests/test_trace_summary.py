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
