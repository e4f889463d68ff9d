"""Decode-step benchmark: batch-1 decode tok/s and achieved HBM GB/s on the Llama-3.2-1B
shape (bf16 weights, fp32 activations, bf16 paged KV cache), seeded synthetic weights.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mie|reference] [--fmt bf16|i8|q4_0]
                [--ctx 128] [--no-cpu-baseline]

One step = one full decode step (embedding gather, 16 layers of fused GEMVs + paged
attention, LM head + argmax) replayed from the captured CUDA graph, token and position
advanced on the device.  The weights (2.47 GB bf16) are far larger than the 129 MB L2,
so nothing is served from L2 between steps.  Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

STEP_PARAMS_BYTES = 112  # sizeof(StepParams): copied host -> device per host-driven step


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="mie", choices=["mie", "reference"])
    ap.add_argument("--fmt", default="bf16", choices=["bf16", "i8", "q4_0"])
    ap.add_argument("--ctx", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=32)
    ap.add_argument("--oracle-steps", type=int, default=3)
    ap.add_argument("--chain", action="store_true", help="one kernel per phase instead of the persistent step")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the dominant kernel (the profiling command)")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class Clocks:
    """Samples nvidia-smi every 200 ms while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                     timeout=5).stdout.strip()
                if out:
                    self.rows.append([c.strip() for c in out.split(",")])
            except Exception:
                pass
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_init(args):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, v: float) -> float:
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle

def oracle_model(shape, ctx: int, n_extra: int):
    """The oracle's model with its K/V cache filled with seeded N(0,1) bf16 values for
    positions < ctx (a synthetic prefill: the step's cost does not depend on the values)."""
    import oracle
    bs = shape.block_size
    n_blocks = (ctx + n_extra + bs - 1) // bs + 1
    om = oracle.Model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * bs)
    kv = om.kv()
    fill = synth.normal(0x4B56, kv.size)
    kv[...] = oracle.to_bf16(fill).reshape(kv.shape)
    return om, np.arange(n_blocks, dtype=np.int32)


def time_oracle(shape, ctx: int, steps: int):
    """Seconds per oracle decode step (single-threaded plain C), over `steps` steps."""
    om, bt = oracle_model(shape, ctx, steps)
    toks = shape.tokens(steps, stream=3)
    t0 = time.perf_counter()
    for i in range(steps):
        om.decode_step(int(toks[i]), ctx + i, bt)
    return (time.perf_counter() - t0) / steps


def run_reference(args, shape):
    rank, world, local, pg = dist_init(args)
    if rank != 0:
        return
    steps = max(1, args.steps)
    om, bt = oracle_model(shape, args.ctx, args.warmup + steps)
    toks = shape.tokens(args.warmup + steps, stream=3)
    for i in range(args.warmup):
        om.decode_step(int(toks[i]), args.ctx + i, bt)
    t0 = time.perf_counter()
    for i in range(steps):
        om.decode_step(int(toks[args.warmup + i]), args.ctx + args.warmup + i, bt)
    dt = (time.perf_counter() - t0) / steps
    v = 1.0 / dt
    line = {"impl": "reference", "metric": "batch-1 decode tok/s", "value": v, "unit": "tok/s",
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate/f32",
            "data": "synthetic (seeded N(0,0.02) weights, uniform tokens)",
            "config": {"workload": f"{shape.name} {args.fmt} decode step, ctx {args.ctx}",
                       "global_batch": 1, "seq_len": args.ctx},
            "cpu_baseline": {"kind": "oracle", "cores": 1, "value": v, "unit": "tok/s",
                             "sample": f"{steps} full decode steps of the oracle (single-threaded C) at ctx "
                                       f"{args.ctx}+, K/V cache prefilled with seeded values"},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def gemv_roofline(torch, mie, n_iter: int = 40):
    """The dominant kernel of the step -- the bf16 GEMV at the gate/up shape
    (16384 x 2048, 42% of the step's weight bytes) -- timed alone with CUDA events on
    its stream, rotating over enough weight copies (> 1 GB) that L2 serves nothing."""
    M, K = 16384, 2048
    copies = 20
    w = torch.empty((copies, M, K), dtype=torch.bfloat16, device="cuda")
    for c in range(copies):
        w[c].copy_(torch.from_numpy(synth.normal(0x525F + c, M * K, std=0.02).reshape(M, K)).to(torch.bfloat16))
    x = torch.from_numpy(synth.normal(0x5260, K)).to(torch.bfloat16).float().cuda()
    y = torch.empty(M, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    for i in range(6):
        mie.mie_gemv_bf16(w[i % copies], x, y, stream=st)
    st.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(n_iter):
        mie.mie_gemv_bf16(w[i % copies], x, y, stream=st)
    e1.record(st)
    e1.synchronize()
    dt = e0.elapsed_time(e1) / 1e3 / n_iter
    algo = M * K * 2 + K * 4 + M * 4
    del w
    torch.cuda.empty_cache()
    return algo, dt, n_iter


def run_mie(args, shape):
    import torch

    rank, world, local, pg = dist_init(args)
    torch.cuda.set_device(local)
    import memory_bound_decode_dequant_gb300 as mie
    from memory_bound_decode_dequant_gb300.workload import build_gpu_model

    bs = shape.block_size
    total = args.ctx + 2 * (args.warmup + args.steps) + args.e2e_steps + 2
    n_blocks = (total + bs - 1) // bs + 1
    max_pos = n_blocks * bs
    stream = torch.cuda.Stream()  # the context's stream: events are recorded on it
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos, stream=stream)
    if args.chain:
        gm.set_step_mode(gm.CHAIN)
    bt_host = synth.permutation(0x4254, n_blocks).astype(np.int32)
    bt = torch.from_numpy(bt_host).cuda()
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    # prefill the context with real decode steps (untimed)
    toks = shape.tokens(args.ctx, stream=rank)
    for pos, t in enumerate(toks):
        gm.decode_step(int(t), pos, bt, logits, am)
    gm.sync()
    launches = gm.launches

    # warm-up, then the timed region: K steps replayed from the graph, token and
    # position advanced on the device; CUDA events on the context's stream
    gm.decode_continue(args.warmup)
    gm.sync()
    barrier(pg)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        t_wall = time.perf_counter()
        e0.record(stream)
        gm.decode_continue(args.steps)
        e1.record(stream)
        e1.synchronize()
        t_wall = time.perf_counter() - t_wall
    gm.sync()
    dt_local = e0.elapsed_time(e1) / 1e3 / args.steps
    barrier(pg)
    dt = max_over_ranks(pg, dt_local)
    ctx_end = args.ctx + args.warmup + args.steps

    # end to end: host token and position in, argmax read back every step
    pos = args.ctx + args.warmup + args.steps
    tok = int(am.item())
    gm.sync()
    barrier(pg)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        gm.decode_step(tok, pos, bt, logits, am)
        tok = int(am.item())  # device -> host read of the step's result (synchronises)
        pos += 1
    gm.sync()
    e2e_dt = max_over_ranks(pg, (time.perf_counter() - t0) / args.e2e_steps)

    # algorithmic bytes of one step: all weights once + the K/V of every position read
    w_bytes = shape.weight_bytes()
    mid_ctx = (args.ctx + 1 + ctx_end) / 2
    kv_bytes = shape.kv_bytes_per_token() * mid_ctx
    step_bytes = w_bytes + kv_bytes
    peak, peak_kind = measured_peaks()

    result = None
    if rank == 0:
        algo, kdt, n_iter = gemv_roofline(torch, mie)
        achieved = algo / kdt / 1e9
        traffic = None
        tp = os.path.join(ROOT, "profiles", "gemv_bf16_16384x2048.traffic.json")
        if os.path.exists(tp):
            with open(tp) as f:
                traffic = json.load(f).get("bytes_per_launch")
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            n = max(1, args.oracle_steps)
            sec = time_oracle(shape, args.ctx, n)
            cpu = {"value": 1.0 / sec, "unit": "tok/s", "cores": 1, "kind": "oracle",
                   "sample": f"{n} full decode steps of the oracle (plain single-threaded C) at ctx {args.ctx}, "
                             f"K/V cache prefilled with seeded values"}
        value = world * 1.0 / dt
        result = {
            "metric": "batch-1 decode tok/s (Llama-3.2-1B shape)",
            "value": value,
            "unit": "tok/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": dt * 1e3,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16 weights, f32 activations/accumulation, bf16 KV",
            "data": "synthetic (seeded N(0,0.02) weights, uniform tokens, prefilled by real decode steps)",
            "config": {"workload": f"{shape.name} {args.fmt} batch-1 decode step",
                       "model": shape.name, "weights": args.fmt, "global_batch": world, "seq_len": args.ctx,
                       "ctx_range": [args.ctx, ctx_end], "parallelism": "replicas" if world > 1 else "single",
                       "l2": "weights 2.47 GB per step >> 129 MB L2: inputs larger than L2",
                       "step_bytes": step_bytes, "step_hbm_gbs": step_bytes / dt / 1e9,
                       "step_frac_of_peak": step_bytes / dt / 1e9 / peak},
            "roofline": {"bound": "hbm", "kernel": "gemv bf16 16384x2048 (gate/up shape)",
                         "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "algorithmic_bytes": algo,
                         "launches_timed": n_iter, "us_per_launch": kdt * 1e6},
            "e2e": {"value": world / e2e_dt, "unit": "tok/s", "h2d_bytes_per_step": STEP_PARAMS_BYTES,
                    "d2h_bytes_per_step": 4},
            "gpu_launches": launches * args.steps,
            "launches_per_step": launches,
            "step_mode": "persistent" if gm.step_mode == 0 else "chain",
            "clocks": clk.summary(),
            "wall_s_timed": t_wall,
            "cpu_baseline": cpu,
        }
        print(json.dumps(result), flush=True)
    gm.close()
    if pg is not None:
        pg.destroy_process_group()
    return result


def main():
    args = parse()
    shape = synth.llama32_1b(args.fmt)
    if args.kernel_only:
        import torch
        import memory_bound_decode_dequant_gb300 as mie
        algo, dt, n = gemv_roofline(torch, mie, n_iter=max(1, args.steps))
        print(json.dumps({"kernel": "gemv bf16 16384x2048", "us_per_launch": dt * 1e6,
                          "achieved_gbs": algo / dt / 1e9, "launches": n}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, shape)
    else:
        run_mie(args, shape)


if __name__ == "__main__":
    main()
