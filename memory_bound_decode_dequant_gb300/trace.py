"""Timeline of the persistent decode step (mie_set_trace), summarised per phase kind.

python -m memory_bound_decode_dequant_gb300.trace [--fmt bf16|i8|q4_0] [--ctx 128] [--stages]

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


def summarise_stages(t: np.ndarray, st: np.ndarray, n_layers: int) -> dict:
    """Per-stage stamps st [ctas, stages, 4] (issued, consumer starts waiting, wait
    returns, consumer done; 0 = not recorded) against the phase stamps t, per phase kind
    averaged over layers and CTAs, microseconds: `lead` = wait start - issue (how early
    the copy was issued), `wait` = wait return - wait start (time the consumer stalled),
    `stalled` = fraction of stages whose wait lasted over 0.1 us, `latency` = wait return
    - issue over the stalled stages (an upper bound on issue -> landing), `math` = done -
    wait return."""
    names = ["qkv", "attn", "o", "gu", "down"] * n_layers + ["head"]
    t = t.astype(np.float64)
    st = st.astype(np.float64)
    agg: dict = {}
    for c in range(st.shape[0]):
        rec = st[c]
        ok = rec[:, 1] > 0
        for p, name in enumerate(names):
            lo, hi = t[p, c, 2], t[p, c, 3]
            sel = ok & (rec[:, 1] >= lo) & (rec[:, 1] <= hi)
            if not np.any(sel):
                continue
            r = rec[sel] / 1e3
            wait = r[:, 2] - r[:, 1]
            stalled = wait > 0.1
            a = agg.setdefault(name, {"lead": [], "wait": [], "stalled": [], "latency": [], "math": [], "n": []})
            a["lead"].append(float(np.mean(r[:, 1] - r[:, 0])))
            a["wait"].append(float(np.mean(wait)))
            a["stalled"].append(float(np.mean(stalled)))
            if np.any(stalled):
                a["latency"].append(float(np.mean(r[stalled, 2] - r[stalled, 0])))
            a["math"].append(float(np.mean(r[:, 3] - r[:, 2])))
            a["n"].append(int(sel.sum()))
    return {k: {kk: round(float(np.mean(v)), 3) if v else None for kk, v in a.items()} for k, a in agg.items()}


def summarise_points(t: np.ndarray, pts: np.ndarray, n_layers: int) -> dict:
    """Points inside each phase (instrumented build), per phase kind, mean over layers
    and CTAs of microseconds since the phase's entry stamp: GEMV phases 0 = input poll
    returned, 1 = RMSNorm done, 2 = input in registers; attention items 3 = inputs
    polled, 4 = first K/V stage landed, 5 = first chunk reduced, 6 = outputs written
    (single-split items).  Points a CTA did not reach are left out."""
    names = ["qkv", "attn", "o", "gu", "down"] * n_layers + ["head"]
    out: dict = {}
    for p, name in enumerate(names):
        e = t[p, :, 0].astype(np.float64)
        for k in range(7):
            v = pts[p, :, k].astype(np.float64)
            ok = v > 0
            if np.any(ok):
                out.setdefault(name, {}).setdefault(k, []).append(float(np.mean(v[ok] - e[ok]) / 1e3))
    return {n: {str(k): round(float(np.mean(v)), 3) for k, v in d.items()} for n, d in out.items()}


def main():
    import torch

    import synth
    from .workload import build_gpu_model

    ap = argparse.ArgumentParser()
    ap.add_argument("--fmt", default="bf16", choices=["bf16", "i8", "q4_0"])
    ap.add_argument("--ctx", type=int, default=128)
    ap.add_argument("--stages", action="store_true",
                    help="also summarise the per-stage stamps (library built with MIE_STAGE_TRACE=1)")
    ap.add_argument("--layers", type=int, default=0, help="truncate the model (0 = all layers)")
    ap.add_argument("--save", default="", help="with --stages: also save the raw stamps (.npz)")
    args = ap.parse_args()
    shape = synth.llama32_1b(args.fmt)
    if args.layers:
        from dataclasses import replace
        shape = replace(shape, n_layers=args.layers)
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
    got = gm.set_trace(True, stages=args.stages)
    buf, stb, sub = got if args.stages else (got, None, None)
    gm.decode_step(int(toks[-1]), args.ctx, bt, logits, am)
    gm.decode_continue(3)
    gm.sync()
    out = summarise(buf.cpu().numpy(), shape.n_layers)
    if args.stages:
        out["stages"] = summarise_stages(buf.cpu().numpy(), stb.cpu().numpy(), shape.n_layers)
        out["points"] = summarise_points(buf.cpu().numpy(), sub.cpu().numpy(), shape.n_layers)
        if args.save:
            np.savez_compressed(args.save, phases=buf.cpu().numpy(), stages=stb.cpu().numpy(), points=sub.cpu().numpy())
    print(json.dumps(out))


if __name__ == "__main__":
    main()
