"""Pins of the byte accounting behind every bandwidth figure, against numbers the pages
print (CPU only; fixtures under tests/golden/, each with its citation).

The roofline's algorithmic bytes come from `synth.ModelShape.weight_bytes`,
`kv_bytes_per_token`, `decode_bytes` and `synth.gemv_bytes`.  The pages print enough of
their own measurements -- weights read per token, tok/s with the matching % of peak,
per-kernel microseconds with GB/s -- that these formulas are fixed up to the printed
rounding.  A wrong byte count per Q4_0 block, an int8 row scale dropped, K/V counted per
query head instead of per KV head, or the K/V term left out of the step each miss at
least one printed figure.
"""
from __future__ import annotations

import json
import os
from dataclasses import replace

import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _within(printed: float, lo: float, hi: float, half_ulp: float) -> bool:
    """Is `printed` a rounding (to +-half_ulp) of some value in [lo, hi]?"""
    return lo - half_ulp <= printed <= hi + half_ulp


DECODE = _load("infer_decode_table.json")
GEMV = _load("infer_gemv_tables.json")
STORAGE = _load("storage_figures.json")


@pytest.mark.parametrize("row", DECODE["rows"], ids=lambda r: r["engine"])
def test_weights_read_per_token(row):
    """Weights read per token, to the page's two decimals in GB."""
    shape = replace(synth.LLAMA32_1B, wfmt=row["wfmt"], head_fmt=row["head_fmt"])
    assert round(shape.weight_bytes() / 1e9, 2) == pytest.approx(row["weights_gb"], abs=1e-9)


@pytest.mark.parametrize("row", DECODE["rows"], ids=lambda r: r["engine"])
def test_step_bytes_reproduce_percent_of_peak(row):
    """(weights + K/V read per step) x tok/s / peak is the printed % of peak at ctx 128:
    128 new tokens after a 128-token prompt."""
    shape = replace(synth.LLAMA32_1B, wfmt=row["wfmt"], head_fmt=row["head_fmt"])
    step = shape.decode_bytes(DECODE["prompt"], DECODE["new_tokens"])
    peak = DECODE["peak_gbs"] * 1e9
    tps = row["tok_s_ctx128"]
    lo = step * (tps - 0.05) / peak * 100
    hi = step * (tps + 0.05) / peak * 100
    # 0.05 pp for the printed rounding plus 0.05 pp of slack for what the page's own
    # accounting may add (activations, the step's argmax)
    assert _within(row["pct_of_peak"], lo, hi, 0.1)


def test_step_bytes_need_the_kv_term():
    """The check above has teeth: leaving the K/V term out, or counting only the prompt,
    misses the printed % of peak for most rows."""
    peak = DECODE["peak_gbs"] * 1e9
    misses_no_kv = misses_prompt_only = 0
    for row in DECODE["rows"]:
        shape = replace(synth.LLAMA32_1B, wfmt=row["wfmt"], head_fmt=row["head_fmt"])
        for ctx, _ in ((0, "no kv"), (DECODE["prompt"], "prompt only")):
            b = shape.weight_bytes() + shape.kv_bytes_per_token() * ctx
            pct = b * row["tok_s_ctx128"] / peak * 100
            if abs(pct - row["pct_of_peak"]) > 0.15:
                if ctx == 0:
                    misses_no_kv += 1
                else:
                    misses_prompt_only += 1
    assert misses_no_kv == len(DECODE["rows"])
    assert misses_prompt_only >= len(DECODE["rows"]) - 1


def test_decode_bytes_mean_context():
    """decode_bytes averages p + 1 attended positions over the steps it covers."""
    s = synth.LLAMA32_1B
    kv = s.kv_bytes_per_token()
    assert s.decode_bytes(0, 1) == s.weight_bytes() + kv  # position 0 attends to itself
    assert s.decode_bytes(128, 128) == s.weight_bytes() + kv * 192.5
    brute = sum(s.weight_bytes() + kv * (p + 1) for p in range(40, 47)) / 7
    assert s.decode_bytes(40, 7) == pytest.approx(brute, rel=1e-15)


@pytest.mark.parametrize("row", GEMV["bf16"], ids=lambda r: r["kernel"])
def test_bf16_gemv_bytes_reproduce_gbs(row):
    M, K, us = row["M"], row["K"], row["us"]
    b = synth.gemv_bytes("bf16", M, K)
    lo, hi = b / ((us + 0.05) * 1e-6) / 1e9, b / ((us - 0.05) * 1e-6) / 1e9
    assert _within(row["gbs"], lo, hi, 0.5)
    pct = row["gbs"] / GEMV["peak_gbs"] * 100  # the page derives % from its GB/s
    assert abs(pct - row["pct"]) <= 0.5 + 1e-9


@pytest.mark.parametrize("row", GEMV["quantized"], ids=lambda r: r["kernel"])
@pytest.mark.parametrize("fmt", ["i8", "q4"])
def test_quantized_gemv_bytes_reproduce_percent(row, fmt):
    """GB/s on the quantized bytes: int8 with a 4-byte scale per row, Q4_0 with 18 bytes
    per 32 weights.  The int4 lm_head reads above the measured copy peak (108 %)."""
    M, K = row["M"], row["K"]
    us = row[f"{fmt}_us"]
    b = synth.gemv_bytes("i8" if fmt == "i8" else "q4_0", M, K)
    peak = GEMV["peak_gbs"] * 1e9
    lo = b / ((us + 0.05) * 1e-6) / peak * 100
    hi = b / ((us - 0.05) * 1e-6) / peak * 100
    assert _within(row[f"{fmt}_pct"], lo, hi, 0.5)


def test_q4_0_block_bytes_are_pinned_by_the_table():
    """The gate_up and lm_head int4 rows fix the block size: 16 bytes of codes with no
    scale, or a 4-byte scale, both miss them."""
    peak = GEMV["peak_gbs"] * 1e9
    for row in GEMV["quantized"]:
        if row["kernel"] not in ("gate_up", "lm_head"):
            continue
        M, K, us = row["M"], row["K"], row["q4_us"]
        for per_block in (16, 20):
            b = M * (K // 32) * per_block + 4 * K + 4 * M
            pct = b / (us * 1e-6) / peak * 100
            assert abs(pct - row["q4_pct"]) > 2


def test_q4_0_bits_per_weight():
    fig = STORAGE["q4_0_bits_per_weight"]
    for m, k in ((1, 32), (7, 4096), (3, 8192)):
        assert synth.matrix_bytes("q4_0", m, k) * 8 / (m * k) == fig["value"]


def test_tinyllama_bf16_weights():
    fig = STORAGE["tinyllama_bf16_weights_gb"]
    s = replace(synth.TINYLLAMA, wfmt="bf16", head_fmt="bf16")
    total = sum(synth.matrix_bytes("bf16", m, k) for _, m, k in s.tensors())
    assert round(total / 1e9, 1) == fig["value"]


def test_qwen2_kv_footprint():
    fig = STORAGE["qwen2_0_5b_kv_bytes_per_token"]
    qwen = synth.ModelShape("qwen2-0.5b", 99, n_layers=24, d_model=896, n_heads=14,
                            n_kv_heads=2, head_dim=64, ffn=4864, vocab=151936, tied=True,
                            rope_theta=1e6, block_size=fig["block_tokens"])
    assert qwen.kv_bytes_per_token() == fig["value"]
