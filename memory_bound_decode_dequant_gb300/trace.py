"""Timeline of the persistent decode step (mie_set_trace), summarised per phase kind.

python -m memory_bound_decode_dequant_gb300.trace [--fmt bf16|i8|q4_0] [--ctx 128]

Builds the Llama-3.2-1B-shape model from the seeded synthetic weights, fills the
context with real decode steps, switches the step to the persistent kernel, records one
step and prints, per phase kind averaged over the layers: the spread over CTAs of the
moment the phase's input arrived, the input staging, the weight streaming (mean and
slowest CTA), the epilogue and the phase's span, in microseconds.
"""
from __future__ import annotations

import argparse
import json

import numpy as np


def summarise(t: np.ndarray, n_layers: int) -> dict:
    """t: [phases, ctas, 5] nanoseconds (points: entry, input arrived, input staged,
    stages consumed, outputs written) -> per-kind means over the layers, microseconds."""
    t = (t.astype(np.float64) - float(t[:, :, 0].min())) / 1e3
    names = ["qkv", "attn", "o", "gu", "down"] * n_layers + ["head"]
    agg: dict = {}
    for p, name in enumerate(names):
        d = {"input_spread": t[p, :, 1].max() - t[p, :, 1].min(),
             "staging": float(np.mean(t[p, :, 2] - t[p, :, 1])),
             "stream_mean": float(np.mean(t[p, :, 3] - t[p, :, 2])),
             "stream_max": float(np.max(t[p, :, 3] - t[p, :, 2])),
             "epilogue": float(np.mean(t[p, :, 4] - t[p, :, 3])),
             "span": t[p, :, 4].max() - t[p, :, 1].min()}
        for k, v in d.items():
            agg.setdefault(name, {}).setdefault(k, []).append(float(v))
    out = {k: {kk: round(float(np.mean(v)), 2) for kk, v in a.items()} for k, a in agg.items()}
    out["step_us"] = round(float(t[:, :, 4].max()), 1)
    return out


def main():
    import torch

    import synth
    from .workload import build_gpu_model

    ap = argparse.ArgumentParser()
    ap.add_argument("--fmt", default="bf16", choices=["bf16", "i8", "q4_0"])
    ap.add_argument("--ctx", type=int, default=128)
    args = ap.parse_args()
    shape = synth.llama32_1b(args.fmt)
    torch.cuda.set_device(0)
    n_blocks = (args.ctx + 8) // shape.block_size + 2
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * shape.block_size)
    gm.set_step_mode(gm.PERSISTENT)
    bt = torch.arange(n_blocks, dtype=torch.int32, device="cuda")
    logits = torch.empty(shape.vocab, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    toks = shape.tokens(args.ctx)
    for pos, tok in enumerate(toks):
        gm.decode_step(int(tok), pos, bt, logits, am)
    gm.sync()
    buf = gm.set_trace(True)
    gm.decode_step(int(toks[-1]), args.ctx, bt, logits, am)
    gm.decode_continue(3)
    gm.sync()
    print(json.dumps(summarise(buf.cpu().numpy(), shape.n_layers)))


if __name__ == "__main__":
    main()
