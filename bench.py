"""Decode-step benchmark: batch-1 decode tok/s and achieved HBM GB/s on the Llama-3.2-1B
shape (bf16 weights, fp32 activations, bf16 paged KV cache), seeded synthetic weights.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mie|reference] [--fmt bf16|i8|q4_0]
                [--ctx 128] [--no-cpu-baseline] [--workload step|slots]

One step = one full decode step (embedding gather, 16 layers of fused GEMVs + paged
attention, LM head + argmax) replayed from the captured CUDA graph, token and position
advanced on the device.  The weights (2.47 GB bf16) are far larger than the 129 MB L2,
so nothing is served from L2 between steps.  Rank 0 prints one JSON line.

--workload sweep: the stateless kernels alone -- GEMVs 3072x2048, 2048x2048, 16384x2048,
2048x8192, 128256x2048 in bf16 / int8 / Q4_0, paged attention (32 q / 8 KV heads, hd 64)
at ctx 512 / 2048 / 8192 over randomly permuted blocks, argmax over 128256 -- each
replayed back to back from a CUDA graph over more than 1 GB of distinct inputs.

--workload slots: the continuous-batching step instead -- 8 slots with contexts drawn
from U[128, 4096], slots 0-3 sharing a refcounted 512-token prefix, block tables in
random physical order from the host block pool, 256 steps with one slot retired and a
256-token request admitted every 32 steps; aggregate tok/s = 8 * steps / time.
"""
from __future__ import annotations

import argparse
import gc
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
SPEC_HBM_GBS = 7900.0  # GB300 HBM3e, nominal; every fraction is also given against it


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="mie", choices=["mie", "reference"])
    ap.add_argument("--fmt", default="bf16", choices=["bf16", "i8", "q4_0", "q4_g64", "q4_g128"],
                    help="layer weights; 4-bit formats keep the tied head in int8 unless --head says otherwise")
    ap.add_argument("--head", default=None, choices=["bf16", "i8", "q4_0", "q4_g64", "q4_g128"],
                    help="format of the tied LM head / embedding (default: bf16 / i8 by --fmt)")
    ap.add_argument("--ctx", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=32)
    ap.add_argument("--oracle-steps", type=int, default=3)
    ap.add_argument("--chain", action="store_true", help="one kernel per phase instead of the persistent step")
    ap.add_argument("--slot-steps", type=int, default=256,
                    help="timed steps of --workload slots (the workload's 256; fewer for profiling)")
    ap.add_argument("--layers", type=int, default=0,
                    help="truncate the model to this many layers (a small case for profiling; 0 = all)")
    ap.add_argument("--workload", default="step", choices=["step", "slots", "sweep", "prefill"],
                    help="step: batch-1 decode (the headline); slots: 8-slot continuous batching; "
                         "sweep: the per-kernel sweep at the Llama-3.2-1B shapes; prefill: the "
                         "2048-token prompt on the tensor cores and its GEMMs")
    ap.add_argument("--gemm", default="",
                    help="with --workload prefill: only the prompt GEMM of this layer shape (qkv, o, "
                         "gate_up, down) at T = 2048, launched --steps times (a profiling case)")
    ap.add_argument("--only", default="",
                    help="sweep: run only the cases whose 'kind:name:fmt' label contains this text "
                         "(e.g. gemv:lm_head:q4_0, attn:512, argmax)")
    ap.add_argument("--sweep-bytes", type=float, default=1.1e9,
                    help="sweep: bytes of distinct inputs each case rotates through")
    ap.add_argument("--sweep-min", type=int, default=20, help="sweep: least number of input copies per case")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the dominant kernel (the profiling command)")
    ap.add_argument("--quick", action="store_true",
                    help="the headline step only: skip the other workloads recorded in the default line")
    ap.add_argument("--decode-steps", type=int, default=128,
                    help="timed decode steps at each context of the per-context table")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_peak() -> float:
    """Dense bf16 tensor TFLOP/s: the driver's burst cuBLAS measurement, else the
    profiling recipe's fallback of 1.9 PFLOP/s."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f).get("bf16_tflops", 1900.0))
    return 1900.0


class NoGC:
    """Pauses Python's cyclic garbage collector inside a timed host loop: collections over
    the objects the earlier workloads of the default line leave behind stalled the host
    between launches and left the GPU idle (measured on GB300: the 8-slot loop ran 1.78 ms
    per step after those workloads, 1.29 ms alone and 1.29 ms after them with the
    collector paused).  No work is skipped; the collector runs once before the loop."""

    def __enter__(self):
        self._on = gc.isenabled()
        gc.collect()
        gc.disable()
        return self

    def __exit__(self, *a):
        if self._on:
            gc.enable()


class Clocks:
    """Samples nvidia-smi every 200 ms while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self._stop = threading.Event()
        self._first = threading.Event()
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
            self._first.set()
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        # the sampler's first query (process start, NVML set-up) ends before the timed
        # region begins; the later ones fall inside it
        self._first.wait(timeout=6)
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


def env_rank() -> tuple[int, int, int]:
    """(RANK, WORLD_SIZE, LOCAL_RANK) as torchrun sets them; (0, 1, 0) when run alone."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(args, backend: str = "nccl"):
    """One process per GPU: each rank runs an independent replica of the step, so the
    process group carries only the start/stop barriers and the max of the ranks' times."""
    rank, world, local = env_rank()
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, v: float) -> float:
    if pg is None:
        return v
    import torch
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
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


def cpu_model() -> str:
    """The host CPU's model string (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def time_oracle(shape, ctx: int, steps: int, threads: int = 1):
    """Seconds per oracle decode step over `steps` steps, on `threads` host threads (the
    oracle spreads GEMV rows and attention heads over them, bit-identically)."""
    import oracle
    om, bt = oracle_model(shape, ctx, steps)
    oracle.set_threads(threads)
    toks = shape.tokens(steps, stream=3)
    try:
        t0 = time.perf_counter()
        for i in range(steps):
            om.decode_step(int(toks[i]), ctx + i, bt)
        return (time.perf_counter() - t0) / steps
    finally:
        oracle.set_threads(1)


def oracle_baseline(shape, ctx: int, steps: int) -> dict:
    """The oracle on all host cores (the reported baseline) and on one core."""
    import oracle
    n = oracle.max_threads()
    sec_all = time_oracle(shape, ctx, steps, threads=n)
    sec_one = time_oracle(shape, ctx, steps, threads=1)
    return {"value": 1.0 / sec_all, "unit": "tok/s", "cores": n, "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{steps} full decode steps of the oracle (plain C, fp64 sums; GEMV rows and attention "
                      f"heads over {n} threads) at ctx {ctx}, K/V cache prefilled with seeded values",
            "single_core": {"value": 1.0 / sec_one, "unit": "tok/s", "cores": 1}}


def run_reference(args, shape):
    if env_rank()[0] != 0:  # under torchrun rank 0 alone times the oracle
        return
    import oracle
    steps = max(1, args.steps)
    om, bt = oracle_model(shape, args.ctx, args.warmup + steps)
    cores = oracle.set_threads(oracle.max_threads())
    toks = shape.tokens(args.warmup + steps, stream=3)
    for i in range(args.warmup):
        om.decode_step(int(toks[i]), args.ctx + i, bt)
    t0 = time.perf_counter()
    for i in range(steps):
        om.decode_step(int(toks[args.warmup + i]), args.ctx + args.warmup + i, bt)
    dt = (time.perf_counter() - t0) / steps
    v = 1.0 / dt
    line = {"impl": "reference", "metric": "batch-1 decode tok/s (Llama-3.2-1B shape)", "value": v, "unit": "tok/s",
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate/f32",
            "data": "synthetic (seeded N(0,0.02) weights, uniform tokens)",
            "config": step_config(args, shape, 1),
            "cpu_baseline": {"kind": "oracle", "cores": cores, "value": v, "unit": "tok/s", "cpu": cpu_model(),
                             "sample": f"{steps} full decode steps of the oracle (plain C, fp64 sums, GEMV rows "
                                       f"and attention heads over {cores} threads) at ctx {args.ctx}+, K/V cache "
                                       f"prefilled with seeded values"},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_slots(args):
    if env_rank()[0] != 0:
        return
    shape = synth.llama32_1b("bf16")
    wl = synth.SlotWorkload()
    cpu = time_oracle_slots(shape, wl)
    v = cpu["value"]
    line = {"impl": "reference", "metric": "continuous-batching decode tok/s (8 slots, Llama-3.2-1B shape bf16)",
            "value": v, "unit": "tok/s", "n_gpus": 1, "steps": 1, "warmup": 0, "ms_per_step": 8e3 / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": "llama-3.2-1b bf16 8-slot continuous-batching step"},
            "cpu_baseline": cpu,
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

CSRC = os.path.join(ROOT, "memory_bound_decode_dequant_gb300", "csrc")


def source_digest(unit: str) -> str:
    """Digest of a translation unit under csrc/ and every local header it includes, with
    comments and layout removed: it changes when the compiled code can, not when a
    comment does."""
    import hashlib
    import re
    seen, order, todo = set(), [], [os.path.normpath(os.path.join(CSRC, unit))]
    while todo:
        path = todo.pop()
        if path in seen:
            continue
        seen.add(path)
        order.append(path)
        with open(path) as f:
            text = f.read()
        for inc in re.findall(r'^\s*#include\s+"([^"]+)"', text, flags=re.M):
            todo.append(os.path.normpath(os.path.join(os.path.dirname(path), inc)))
    h = hashlib.sha256()
    for path in sorted(order):
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(os.path.relpath(path, ROOT).encode() + b"\0" + " ".join(text.split()).encode() + b"\0")
    return h.hexdigest()[:16]


def read_traffic(name: str):
    """DRAM bytes per launch of a kernel from its ncu record under profiles/, or None when
    there is no record or the kernel's source has changed since the counters were taken."""
    tp = os.path.join(ROOT, "profiles", f"{name}.traffic.json")
    if not os.path.exists(tp):
        return None
    with open(tp) as f:
        rec = json.load(f)
    unit, digest = rec.get("translation_unit"), rec.get("source_digest")
    if not unit or not digest or source_digest(unit) != digest:
        return None
    return rec.get("bytes_per_launch")


def gemv_roofline(torch, mie, n_iter: int = 40):
    """The dominant kernel of the step -- the bf16 GEMV at the gate/up shape
    (16384 x 2048, 42% of the step's weight bytes) -- timed alone with CUDA events on
    its stream: n_iter back-to-back launches captured in one CUDA graph (so no host
    launch gap sits between them), rotating over enough weight copies (> 1 GB) that L2
    serves nothing; the median of 5 replays."""
    M, K = 16384, 2048
    copies = 20
    w = torch.empty((copies, M, K), dtype=torch.bfloat16, device="cuda")
    for c in range(copies):
        w[c].copy_(torch.from_numpy(synth.normal(0x525F + c, M * K, std=0.02).reshape(M, K)).to(torch.bfloat16))
    x = torch.from_numpy(synth.normal(0x5260, K)).to(torch.bfloat16).float().cuda()
    y = torch.empty(M, dtype=torch.float32, device="cuda")
    dt = graph_time(torch, [(lambda st, i=i: mie.mie_gemv_bf16(w[i % copies], x, y, stream=st))
                            for i in range(n_iter)])
    algo = synth.gemv_bytes("bf16", M, K)
    del w
    torch.cuda.empty_cache()
    return algo, dt, n_iter


def read_probe(torch, mie, gib: int = 4) -> dict:
    """The read-only streaming peak of this GPU: mie_hbm_read_probe over a `gib` GiB
    buffer (31 x L2 at 4 GiB), 16- and 32-byte loads at 1, 2 and 4 CTAs per SM, the
    best median of 10 back-to-back launches."""
    buf = torch.empty((gib << 28,), dtype=torch.int32, device="cuda")
    buf.fill_(0x5A5A5A5A)
    nbytes = buf.numel() * 4
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    runs = []
    for load in (16, 32):
        for bps in (1, 2, 4):
            for _ in range(3):
                mie.mie_hbm_read_probe(buf, out, load, bps, stream=st)
            times = []
            for _ in range(3):  # 10 back-to-back launches between one pair of events
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                for _ in range(10):
                    mie.mie_hbm_read_probe(buf, out, load, bps, stream=st)
                e1.record(st)
                e1.synchronize()
                times.append(e0.elapsed_time(e1) / 1e3 / 10)
            runs.append({"load_bytes": load, "blocks_per_sm": bps, "gbs": nbytes / statistics.median(times) / 1e9})
    del buf
    torch.cuda.empty_cache()
    best = max(runs, key=lambda r: r["gbs"])
    return {"gbs": best["gbs"], "best": best, "bytes": nbytes, "runs": runs,
            "method": f"mie_hbm_read_probe over {gib} GiB; per setting the median of 3 timings of 10 "
                      f"back-to-back launches"}


def contexts_table(torch, gm, stream, shape, bt, logits, am, pos: int, tok: int, ctxs, steps: int, peak: float,
                   read_peak: float | None) -> tuple[list, int, int]:
    """For each context in order: real greedy decode steps (untimed) bring the sequence
    to that context, then `steps` steps replayed from the graph are timed with events on
    the context's stream.  Returns the rows and the position and token reached."""
    rows = []
    for ctx in ctxs:
        if ctx <= pos:
            continue
        gm.decode_step(tok, pos, bt, logits, am)  # the step at pos; the graph advances from there
        gm.decode_continue(ctx - pos - 1)  # the next step writes position ctx
        gm.sync()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gm.decode_continue(steps)
        e1.record(stream)
        e1.synchronize()
        gm.sync()
        dt = e0.elapsed_time(e1) / 1e3 / steps
        b = shape.decode_bytes(ctx, steps)
        row = {"ctx": ctx, "steps": steps, "tok_s": 1.0 / dt, "ms_per_step": dt * 1e3, "step_bytes": b,
               "gbs": b / dt / 1e9, "frac_of_peak": b / dt / 1e9 / peak}
        if read_peak:
            row["frac_of_read_probe"] = b / dt / 1e9 / read_peak
        rows.append(row)
        pos = ctx + steps
        with torch.cuda.stream(stream):
            tok = int(am.item())
    return rows, pos, tok


def sampled_steps(torch, gm, stream, bt, logits, am, pos: int, tok: int, steps: int) -> dict:
    """The same step with the next token drawn by temperature 0.6 / top-k 40 / top-p 0.9
    sampling inside its graph (mie_set_sampling), timed like the greedy step."""
    T, k, p = 0.6, 40, 0.9
    gm.set_sampling(T, k, p, 0x5A4D)
    gm.decode_step(tok, pos, bt, logits, am)
    gm.decode_continue(3)
    gm.sync()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    gm.decode_continue(steps)
    e1.record(stream)
    e1.synchronize()
    gm.sync()
    dt = e0.elapsed_time(e1) / 1e3 / steps
    gm.set_sampling(0.0)
    return {"temperature": T, "top_k": k, "top_p": p, "ctx": pos + 4, "steps": steps, "tok_s": 1.0 / dt,
            "ms_per_step": dt * 1e3, "launches_per_step": gm.launches}


GEMM_SHAPES = [("qkv", 3072, 2048), ("o", 2048, 2048), ("gate_up", 16384, 2048), ("down", 2048, 8192)]


def prefill_measure(torch, bf16_peak: float, n_prompt: int = 2048, chunk: int = 2048) -> dict:
    """Prompt prefill on the tensor cores (mie_prefill) at the Llama-3.2-1B shape with bf16
    weights: an n_prompt-token prompt (one chunk of up to 2048 positions), timed with
    events on the model's stream; and the tcgen05 GEMM alone at the four layer shapes for
    one chunk (three activation planes: three MMAs per product), graph-timed over copies
    of the weights larger than L2, against the measured bf16 tensor peak."""
    from memory_bound_decode_dequant_gb300.workload import build_gpu_model
    import memory_bound_decode_dequant_gb300 as mie
    shape = synth.llama32_1b("bf16")
    bs = shape.block_size
    n_blocks = (n_prompt + bs - 1) // bs + 2
    stream = torch.cuda.Stream()
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * bs, stream=stream)
    bt = torch.from_numpy(synth.permutation(0x5046, n_blocks).astype(np.int32)).cuda()
    toks = [int(t) for t in shape.tokens(n_prompt, stream=14)]
    gm.prefill(toks[:64], 0, bt)  # buffers
    gm.sync()
    times = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gm.prefill(toks, 0, bt)
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    gm.sync()
    gm.close()
    del gm
    dt = statistics.median(times)
    L, d, f = shape.n_layers, shape.d_model, shape.ffn
    na = shape.n_heads * shape.head_dim
    qkv = shape.qkv_rows * d
    per_tok = 2 * (L * qkv + (L - 1) * (d * na + 2 * f * d + d * f))  # the last layer stops after K/V
    attn = (L - 1) * 4 * na * n_prompt * (n_prompt + 1) / 2  # causal QK^T and PV
    flops = per_tok * n_prompt + attn
    out = {"workload": f"llama-3.2-1b bf16 prompt prefill, {n_prompt} tokens", "chunk": chunk,
           "ms": dt * 1e3, "tok_s": n_prompt / dt, "useful_tflops": flops / dt / 1e12,
           "kernels": "tcgen05 GEMM (TMA, TMEM accumulators, 3 bf16 activation planes) + mma.sync flash attention",
           "method": "CUDA events on the model's stream around mie_prefill, median of 3"}
    gemms = []
    for name, N, K in GEMM_SHAPES:
        nbytes = N * K * 2
        copies = max(2, int(np.ceil(300e6 / nbytes)))
        Ws = [torch.randn(N, K, device="cuda").mul_(0.02).to(torch.bfloat16) for _ in range(copies)]
        x = torch.randn(chunk, K, device="cuda")
        planes = mie.mie_split_bf16(x)
        y = torch.empty(chunk, N, device="cuda")
        n_launch = 4 * copies
        t = graph_time(torch, [lambda st, W=Ws[i % copies]: mie.mie_gemm_bf16(W, planes, y, stream=st)
                               for i in range(n_launch)])
        useful = 2.0 * N * K * chunk / t / 1e12
        tensor = 3 * useful
        gemms.append({"gemm": name, "N": N, "K": K, "T": chunk, "us": t * 1e6, "useful_tflops": useful,
                      "tensor_tflops": tensor, "frac_of_bf16_peak": tensor / bf16_peak,
                      "weight_copies": copies})
        del Ws, x, planes, y
    torch.cuda.empty_cache()
    top = max(gemms, key=lambda g: g["us"])
    out["gemm"] = gemms
    out["roofline"] = {"bound": "tensor", "kernel": f"gemm_tc_kernel ({top['gemm']} {top['N']}x{top['K']}, "
                                                    f"T = {chunk})",
                       "achieved": top["tensor_tflops"], "peak": bf16_peak, "peak_kind": "measured (burst)",
                       "unit": "TFLOP/s", "frac": top["tensor_tflops"] / bf16_peak,
                       "note": "tensor-pipe rate: three bf16 MMAs per product (hi, mid, lo planes)"}
    return out


def batched_passes(torch, n_spec_prompt: int = 256, n_new: int = 128) -> dict:
    """Llama-3.2-1B bf16 through the few-slot kernels: greedy generation (mie_generate)
    after a prompt that repeats a 64-token pattern, with prompt-lookup speculation (up to
    3 guesses a pass) and without (the two give the same tokens), and the cost of one
    verify pass over k positions against k passes of one."""
    from memory_bound_decode_dequant_gb300.workload import build_gpu_model
    shape = synth.llama32_1b("bf16")
    bs = shape.block_size
    n_blocks = (n_spec_prompt + n_new + bs - 1) // bs + 2
    stream = torch.cuda.Stream()
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * bs, max_slots=8, stream=stream)
    bt = torch.from_numpy(synth.permutation(0x5045, n_blocks).astype(np.int32)).cuda()
    out = {"model": "llama-3.2-1b bf16", "kernels": "few-slot step (mma.sync, bf16 hi + lo inputs)"}
    gm.generate([int(t) for t in shape.tokens(40, stream=11)], 1, bt, 1)  # captures the few-slot graph
    torch.cuda.synchronize()
    pattern = [int(t) for t in shape.tokens(64, stream=12)]
    rep = (pattern * (n_spec_prompt // 64 + 1))[:n_spec_prompt]
    res = {}
    for spec in (1, 4):
        gm.generate(rep, 1, bt, spec)  # the prompt's K/V, untimed
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        toks, st = gm.generate(rep, n_new, bt, spec)
        res[spec] = (toks, st, time.perf_counter() - t0)
    # the payoff the lookup relies on: one pass over k positions against k passes of one
    per_pass = {}
    for k in (1, 2, 4, 8):
        toks = [int(t) for t in shape.tokens(k, stream=13)]
        for i in range(3):
            gm.verify_step(toks, 64 + 8 * i, bt)
        gm.sync()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_rep = 24
        e0.record(stream)
        for i in range(n_rep):
            gm.verify_step(toks, 64 + 8 * (i % 8), bt)
        e1.record(stream)
        e1.synchronize()
        gm.sync()
        per_pass[k] = e0.elapsed_time(e1) / 1e3 / n_rep
    out["pass_cost"] = {str(k): {"ms_per_pass": t * 1e3, "k_single_passes_over_one_pass": k * per_pass[1] / t}
                        for k, t in per_pass.items()}
    gm.close()
    del gm
    torch.cuda.empty_cache()
    same = bool(np.array_equal(res[1][0], res[4][0]))
    out["speculative"] = {"prompt": f"{n_spec_prompt} tokens repeating a 64-token pattern", "new_tokens": n_new,
                          "plain": {"seconds": res[1][2], **res[1][1]},
                          "spec_max_4": {"seconds": res[4][2], **res[4][1]},
                          "same_tokens": same,
                          "note": "wall time includes the prompt's prefill passes"}
    return out


def model_contexts(torch, shape, ctxs, steps: int, peak: float, read_peak: float | None, label: str) -> dict:
    """A fresh context for `shape`, prefilled from position 0 by real decode steps,
    timed at each context of ctxs (contexts_table)."""
    from memory_bound_decode_dequant_gb300.workload import build_gpu_model
    bs = shape.block_size
    n_blocks = (max(ctxs) + steps + bs - 1) // bs + 2
    stream = torch.cuda.Stream()
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * bs, stream=stream)
    bt = torch.from_numpy(synth.permutation(0x4254, n_blocks).astype(np.int32)).cuda()
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    rows, _, _ = contexts_table(torch, gm, stream, shape, bt, logits, am, 0, int(shape.tokens(1)[0]), ctxs, steps,
                                peak, read_peak)
    out = {"workload": label, "weights": shape.wfmt, "head": shape.head_fmt, "weight_bytes": shape.weight_bytes(),
           "step_mode": "persistent" if gm.step_mode == 0 else "chain", "contexts": rows}
    gm.close()
    del gm
    torch.cuda.empty_cache()
    return out


def run_mie(args, shape):
    import torch

    rank, world, local, pg = dist_init(args)
    torch.cuda.set_device(local)
    import memory_bound_decode_dequant_gb300 as mie
    from memory_bound_decode_dequant_gb300.workload import build_gpu_model

    bs = shape.block_size
    ctxs = [c for c in CONTEXTS[shape.name] if c > args.ctx] if not args.quick else []
    total = max([args.ctx + 2 * (args.warmup + args.steps) + args.e2e_steps + 2] +
                [c + 2 * args.decode_steps + 16 for c in ctxs])  # room for the sampled steps after the last
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

    # end to end through mie_decode_step_sync: host token and position in (a pinned upload
    # of the step parameters), the next token read back to the host every step
    pos = args.ctx + args.warmup + args.steps
    with torch.cuda.stream(stream):
        tok = int(am.item())
    gm.sync()
    barrier(pg)
    with NoGC():
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            tok = gm.decode_step_sync(tok, pos, bt, logits)
            pos += 1
        gm.sync()
        e2e_dt_local = (time.perf_counter() - t0) / args.e2e_steps
    e2e_dt = max_over_ranks(pg, e2e_dt_local)

    # algorithmic bytes of one step: all weights once + the K/V of every position read
    step_bytes = shape.decode_bytes(args.ctx + args.warmup, args.steps)  # the timed steps
    peak, peak_kind = measured_peaks()
    extras = {}
    if rank == 0 and world == 1 and not args.quick:
        extras["read_probe"] = guarded(lambda: read_probe(torch, mie))
    read_peak = (extras.get("read_probe") or {}).get("gbs")
    if ctxs:  # the longer contexts of the same sequence, on the same context
        head = {"ctx": args.ctx, "steps": args.steps, "tok_s": 1.0 / dt, "ms_per_step": dt * 1e3,
                "step_bytes": step_bytes, "gbs": step_bytes / dt / 1e9, "frac_of_peak": step_bytes / dt / 1e9 / peak}
        if read_peak:
            head["frac_of_read_probe"] = step_bytes / dt / 1e9 / read_peak
        rows, pos, tok = contexts_table(torch, gm, stream, shape, bt, logits, am, pos, tok, ctxs, args.decode_steps,
                                        peak, read_peak)
        extras["contexts"] = [head] + rows
        extras["sampled"] = guarded(lambda: sampled_steps(torch, gm, stream, bt, logits, am, pos, tok,
                                                          args.decode_steps))

    result = None
    step_mode = "persistent" if gm.step_mode == 0 else "chain"
    if rank == 0:
        algo, kdt, n_iter = gemv_roofline(torch, mie)
        achieved = algo / kdt / 1e9
        gemv_roof = {"bound": "hbm", "kernel": "gemv bf16 16384x2048 (gate/up shape), standalone",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "frac_of_spec": achieved / SPEC_HBM_GBS,
                     "traffic": read_traffic("gemv_bf16_16384x2048"),
                     "algorithmic_bytes": algo, "launches_timed": n_iter, "us_per_launch": kdt * 1e6,
                     "method": "40 back-to-back launches in one CUDA graph, median of 5 replays"}
        if gm.step_mode == 0:
            # the persistent step is the step's only launch: its duration is the step time
            # measured above with events on its stream
            ach = step_bytes / dt / 1e9
            roof = {"bound": "hbm", "kernel": "persistent_step (one launch = one decode step)",
                    "achieved": ach, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": ach / peak,
                    "frac_of_spec": ach / SPEC_HBM_GBS,
                    "traffic": read_traffic(f"persistent_step_llama32_{args.fmt}"),
                    "algorithmic_bytes": step_bytes, "launches_timed": args.steps, "us_per_launch": dt * 1e6}
        else:
            roof = gemv_roof
        for r in (roof, gemv_roof):
            if read_peak:
                r["read_probe_gbs"] = read_peak
                r["frac_of_read_probe"] = r["achieved"] / read_peak
    gm.close()
    del gm
    torch.cuda.empty_cache()
    if rank == 0:
        if world == 1 and not args.quick:
            # the other workloads of the decode-step family, each recorded in this line
            # the other storage variants of the same model (the infer page's decode table):
            # int8, int4 g32 with an int8 head, int4 g32, int4 g128, int4 g128 with an int8 head
            variants = [("i8", None), ("q4_0", None), ("q4_0", "q4_0"), ("q4_g128", "q4_g128"),
                        ("q4_g128", "i8"), ("bf16", None)]
            for f, h in variants:
                sh = synth.llama32_1b(f, h)
                if (sh.wfmt, sh.head_fmt) == (shape.wfmt, shape.head_fmt):
                    continue
                key = f"contexts_{f}" + (f"_head_{sh.head_fmt}" if h else "")
                extras[key] = guarded(lambda sh=sh: model_contexts(
                    torch, sh, CONTEXTS["llama-3.2-1b"], args.decode_steps, peak, read_peak,
                    f"llama-3.2-1b {sh.wfmt} layers, {sh.head_fmt} head, batch-1 decode"))
            extras["tinyllama_q4_0"] = guarded(lambda: model_contexts(
                torch, synth.TINYLLAMA, CONTEXTS["tinyllama-1.1b"], args.decode_steps, peak, read_peak,
                "tinyllama-1.1b q4_0 (bf16 GEMV inputs) batch-1 decode"))
            extras["slots"] = guarded(lambda: slots_summary(measure_slots(args, torch)))
            extras["batched_passes"] = guarded(lambda: batched_passes(torch))
            extras["prefill"] = guarded(lambda: prefill_measure(torch, measured_bf16_peak()))
            extras["kernel_sweep"] = guarded(lambda: measure_sweep(args, clocks=False))
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = oracle_baseline(shape, args.ctx, max(1, args.oracle_steps))
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
            "config": step_config(args, shape, world),
            "step_hbm": {"step_bytes": step_bytes, "gbs": step_bytes / dt / 1e9,
                         "frac_of_peak": step_bytes / dt / 1e9 / peak,
                         "frac_of_spec": step_bytes / dt / 1e9 / SPEC_HBM_GBS,
                         "frac_of_read_probe": (step_bytes / dt / 1e9 / read_peak) if read_peak else None},
            "roofline": roof,
            "gemv_roofline": gemv_roof,
            "e2e": {"value": world / e2e_dt, "unit": "tok/s", "h2d_bytes_per_step": STEP_PARAMS_BYTES,
                    "d2h_bytes_per_step": 4},
            "gpu_launches": launches * args.steps,
            "launches_per_step": launches,
            "step_mode": step_mode,
            "clocks": clk.summary(),
            "wall_s_timed": t_wall,
            "cpu_baseline": cpu,
        }
        result.update(extras)
        print(json.dumps(result), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return result


def step_config(args, shape, world: int) -> dict:
    """The workload of the batch-1 line, the same dict in both arms."""
    return {"workload": f"{shape.name} {args.fmt}" + (f" ({shape.head_fmt} head)" if args.head else "")
                        + " batch-1 decode step"
                        + (f" ({shape.n_layers} layers, profiling case)" if args.layers else ""),
            "model": shape.name, "weights": args.fmt, "head": shape.head_fmt, "global_batch": world,
            "seq_len": args.ctx,
            "ctx_range": [args.ctx, args.ctx + args.warmup + args.steps],
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "weights 2.47 GB per step >> 129 MB L2: inputs larger than L2",
            "step_bytes": shape.decode_bytes(args.ctx + args.warmup, args.steps)}


def guarded(fn):
    """Runs one of the extra workloads of the default line; a failure is reported in its
    key instead of losing the headline."""
    try:
        return fn()
    except Exception as e:  # noqa: BLE001 -- the line must still be printed
        import traceback
        return {"error": f"{type(e).__name__}: {e}", "where": traceback.format_exc().splitlines()[-3:]}


# the contexts each workload is quoted at (the decode tables of the pages: Llama-3.2-1B at
# 128 / 512 / 2048, TinyLlama at 50 / 500 / 1500)
CONTEXTS = {"llama-3.2-1b": [128, 512, 2048], "tinyllama-1.1b": [50, 500, 1500]}


# ----------------------------------------------------------------------------- few-slot step

def slot_tables(pool, wl, n_blocks: int, bs: int, max_blocks: int, seed: int):
    """The context's host block pool with its free list shuffled (tables in random
    physical order), the shared prefix of slots 0..shared_slots-1 (refcount
    shared_slots) and each slot's blocks for its context plus the steps it runs."""
    ids = [pool.alloc() for _ in range(n_blocks)]
    for i in synth.permutation(seed, n_blocks):
        pool.decref(ids[int(i)])
    tables = np.zeros((wl.n_slots, max_blocks), np.int32)
    n_prefix = wl.shared_prefix // bs
    prefix = [pool.alloc() for _ in range(n_prefix)]
    for s in range(wl.n_slots):
        nb = (int(wl.ctx[s]) + wl.steps + bs - 1) // bs
        for b in range(nb):
            if s < wl.shared_slots and b < n_prefix:
                tables[s, b] = prefix[b]
                if s > 0:
                    pool.incref(prefix[b])
            else:
                tables[s, b] = pool.alloc()
    assert all(pool.refcount(b) == wl.shared_slots for b in prefix)
    return pool, tables, prefix


def run_slots(args):
    import torch

    rank, world, local, pg = dist_init(args)
    torch.cuda.set_device(local)
    line = measure_slots(args, torch, rank=rank, world=world, local=local,
                         with_cpu=rank == 0 and not args.no_cpu_baseline and world == 1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def slots_summary(line: dict) -> dict:
    """The few-slot workload's figures as one key of the default line."""
    keep = ("metric", "value", "unit", "ms_per_step", "steps", "dtype", "config", "roofline", "e2e",
            "launches_per_step", "clocks")
    return {k: line[k] for k in keep if k in line}


def measure_slots(args, torch, rank: int = 0, world: int = 1, local: int | None = None,
                  with_cpu: bool = False) -> dict:
    """The 8-slot continuous-batching workload (--workload slots); returns its line."""
    from memory_bound_decode_dequant_gb300.workload import build_gpu_model
    if local is None:
        local = torch.cuda.current_device()

    shape = synth.llama32_1b("bf16")
    if args.layers:  # a truncated model for profiling captures
        from dataclasses import replace as _replace
        shape = _replace(shape, n_layers=args.layers)
    wl = synth.SlotWorkload(steps=args.slot_steps)
    bs = shape.block_size
    S = wl.n_slots
    max_ctx = int(wl.ctx.max()) + wl.steps + args.warmup + 1
    max_blocks = (max_ctx + bs - 1) // bs + 1
    n_blocks = S * max_blocks + 64
    stream = torch.cuda.Stream()
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_blocks * bs, max_slots=S, stream=stream)
    # synthetic prefilled cache: every block holds seeded N(0,1) bf16 values
    kv = gm.kv()
    gen = torch.Generator(device="cuda").manual_seed(0x4B56)
    flat = kv.view(-1)
    for i in range(0, flat.numel(), 1 << 26):
        n = min(1 << 26, flat.numel() - i)
        flat[i:i + n].copy_(torch.randn(n, generator=gen, device="cuda").to(torch.bfloat16).view(torch.int16))
    pool, tables, prefix = slot_tables(gm.pool, wl, n_blocks, bs, max_blocks, seed=0x534C)
    tdev = torch.from_numpy(tables).cuda()
    logits = None
    am = torch.empty(S, dtype=torch.int32, device="cuda")
    toks = shape.tokens(S * (wl.steps + args.warmup + 64), stream=7).astype(np.int32).reshape(-1, S)
    pos = wl.ctx.astype(np.int32).copy()
    for i in range(args.warmup):
        gm.decode_step_slots(toks[i], pos, tdev, logits, am)
        pos += 1
    gm.sync()
    torch.cuda.synchronize()

    # timed: wl.steps batched steps through the public call; every admit_every steps the
    # host retires one slot (round robin), releases its blocks to the pool and admits a
    # new admit_len-token request into fresh blocks (its K/V already holds seeded values)
    kv_tokens = 0
    retired = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk, NoGC():
        t_wall = time.perf_counter()
        e0.record(stream)
        for i in range(wl.steps):
            if i > 0 and i % wl.admit_every == 0:
                s = retired % S
                retired += 1
                nb = (int(pos[s]) + bs) // bs
                for b in tables[s, :nb]:
                    pool.decref(int(b))
                new_len = wl.admit_len
                need = (new_len + wl.steps + bs - 1) // bs
                row = np.zeros(max_blocks, np.int32)
                for b in range(need):
                    row[b] = pool.alloc()
                tables[s] = row
                with torch.cuda.stream(stream):  # ordered before the next step on its stream
                    tdev[s].copy_(torch.from_numpy(row))
                pos[s] = new_len
            gm.decode_step_slots(toks[args.warmup + i], pos, tdev, logits, am)
            kv_tokens += int(pos.sum()) + S
            pos += 1
        e1.record(stream)
        e1.synchronize()
        t_wall = time.perf_counter() - t_wall
    gm.sync()
    dt = e0.elapsed_time(e1) / 1e3 / wl.steps
    # end to end: the same call with the argmax read back every step
    e2e_steps = 16
    with NoGC():
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            gm.decode_step_slots(toks[args.warmup + wl.steps + i], pos, tdev, logits, am)
            with torch.cuda.stream(stream):  # the read is ordered after the step on its stream
                _ = am.cpu()  # device -> host read of the step's results (synchronises)
            pos += 1
        e2e_dt = (time.perf_counter() - t0) / e2e_steps
    gm.sync()
    w_bytes = shape.weight_bytes()
    kv_bytes = shape.kv_bytes_per_token() * kv_tokens / wl.steps
    step_bytes = w_bytes + kv_bytes
    peak, peak_kind = measured_peaks()
    cpu = time_oracle_slots(shape, wl) if with_cpu else None
    line = None
    if rank == 0:
        ach = step_bytes / dt / 1e9
        line = {
            "metric": "continuous-batching decode tok/s (8 slots, Llama-3.2-1B shape bf16)",
            "value": world * S / dt, "unit": "tok/s", "n_gpus": world, "steps": wl.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 weights, bf16 hi+lo inputs on tensor cores with f32 accumulation, bf16 KV",
            "data": "synthetic (seeded N(0,0.02) weights, seeded N(0,1) K/V cache, uniform tokens)",
            "config": {"workload": "llama-3.2-1b bf16 8-slot continuous-batching step", "global_batch": S * world,
                       "ctx_initial": [int(c) for c in wl.ctx], "shared_prefix": wl.shared_prefix,
                       "shared_slots": wl.shared_slots, "admit_every": wl.admit_every, "admit_len": wl.admit_len,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "weights 2.47 GB per step >> 129 MB L2: inputs larger than L2",
                       "step_bytes": step_bytes, "kv_bytes_per_step": kv_bytes},
            "roofline": {"bound": "hbm", "kernel": "whole few-slot step (kernel chain in one graph)",
                         "achieved": ach, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": ach / peak, "frac_of_spec": ach / SPEC_HBM_GBS, "traffic": None,
                         "algorithmic_bytes": step_bytes,
                         "us_per_step": dt * 1e6},
            "e2e": {"value": world * S / e2e_dt, "unit": "tok/s", "h2d_bytes_per_step": STEP_PARAMS_BYTES,
                    "d2h_bytes_per_step": 4 * S},
            "gpu_launches": gm.slot_launches * wl.steps, "launches_per_step": gm.slot_launches,
            "clocks": clk.summary(), "wall_s_timed": t_wall, "cpu_baseline": cpu,
        }
    gm.close()
    del gm
    torch.cuda.empty_cache()
    return line


def time_oracle_slots(shape, wl):
    """The oracle's batched step (independent single-slot steps) on a bounded sample:
    two of the eight slots, at their contexts, K/V prefilled with seeded values."""
    import oracle
    bs = shape.block_size
    sample = [0, S_last] if (S_last := wl.n_slots - 1) else [0]
    ctxs = [int(wl.ctx[s]) for s in sample]
    need = sum((c + 1 + bs - 1) // bs for c in ctxs) + 1
    om = oracle.Model(shape, n_kv_blocks=need, max_pos=(max(ctxs) + bs) // bs * bs + bs)
    kv = om.kv()
    kv[...] = oracle.to_bf16(synth.normal(0x4B56, kv.size)).reshape(kv.shape)
    toks = shape.tokens(len(sample), stream=9)
    t0 = time.perf_counter()
    off = 0
    for j, c in enumerate(ctxs):
        nb = (c + 1 + bs - 1) // bs
        bt = np.arange(off, off + nb, dtype=np.int32)
        off += nb
        om.decode_step(int(toks[j]), c, bt)
    sec_per_slot = (time.perf_counter() - t0) / len(sample)
    return {"value": 1.0 / sec_per_slot, "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": f"slots {sample} of the 8 (contexts {ctxs}) through the oracle's single-slot step, "
                      f"which defines its batched step; plain single-threaded C, K/V seeded"}


# ----------------------------------------------------------------------------- per-kernel sweep

def graph_time(torch, launches, reps: int = 5):
    """Seconds per launch of a list of closures replayed from one CUDA graph (median)."""
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for f in launches[:3]:
            f(st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for f in launches:
            f(st)
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        with torch.cuda.stream(st):
            g.replay()
        e1.record(st)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3 / len(launches))
    return statistics.median(times)


def run_sweep(args):
    import torch
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    print(json.dumps(measure_sweep(args)), flush=True)


def measure_sweep(args, clocks: bool = True) -> dict:
    """The per-kernel sweep (--workload sweep); returns its record."""
    import contextlib
    import torch
    import memory_bound_decode_dequant_gb300 as mie

    peak, peak_kind = measured_peaks()
    gen = torch.Generator(device="cuda").manual_seed(synth.SWEEP_SEED)
    total, least = args.sweep_bytes, args.sweep_min
    want = lambda label: args.only in label
    out = {"metric": "per-kernel sweep (Llama-3.2-1B decode shapes)", "unit": "us / GB/s per launch",
           "peak_gbs": peak, "peak_kind": peak_kind, "gemv": [], "attention": [], "argmax": None,
           "method": "graph of back-to-back launches over > 1 GB of distinct inputs; median of 5 replays"}
    clk = Clocks(int(os.environ.get("LOCAL_RANK", 0))) if clocks else None
    with clk or contextlib.nullcontext():
        for name, M, K in synth.SWEEP_GEMV:
            if not any(want(f"gemv:{name}:{f}") for f in ("bf16", "i8", "q4_0")):
                continue
            w = torch.randn((M, K), generator=gen, device="cuda") * 0.02
            x = torch.randn(K, generator=gen, device="cuda").to(torch.bfloat16).float()
            y = torch.empty(M, dtype=torch.float32, device="cuda")
            for fmt in ("bf16", "i8", "q4_0"):
                if not want(f"gemv:{name}:{fmt}"):
                    continue
                if fmt == "bf16":
                    one = (mie.mie_convert_bf16(w),)
                    nbytes = synth.matrix_bytes("bf16", M, K)
                    call = lambda a, st: mie.mie_gemv_bf16(a[0], x, y, stream=st)
                elif fmt == "i8":
                    one = mie.mie_quantize_i8(w)
                    nbytes = synth.matrix_bytes("i8", M, K)
                    call = lambda a, st: mie.mie_gemv_i8(a[0], a[1], x, y, stream=st)
                else:
                    one = (mie.mie_q4_0_pack(mie.mie_quantize_q4_0(w), M, K),)
                    nbytes = synth.matrix_bytes("q4_0", M, K)
                    call = lambda a, st: mie.mie_gemv_q4_0(a[0], x, M, K, y, stream=st)
                n = max(least, int(total // nbytes) + 1)
                copies = [one] + [tuple(t.clone() for t in one) for _ in range(n - 1)]
                dt = graph_time(torch, [(lambda st, a=a: call(a, st)) for a in copies])
                algo = synth.gemv_bytes(fmt, M, K)
                out["gemv"].append({"shape": [M, K], "name": name, "fmt": fmt, "us": dt * 1e6,
                                    "gbs": algo / dt / 1e9, "frac": algo / dt / 1e9 / peak, "launches": n})
                del copies, one
                torch.cuda.empty_cache()
            del w
        Hq, Hkv, hd, bs = 32, 8, 64, 16
        for ctx in synth.SWEEP_ATTN_CTX:
            if not want(f"attn:{ctx}"):
                continue
            nblk = (ctx + bs - 1) // bs
            per_call = ctx * Hkv * hd * 2 * 2
            n = max(least, int(total // per_call) + 1)
            pool_blocks = nblk * n
            k_pool = torch.randn((pool_blocks, Hkv, bs, hd), generator=gen, device="cuda").to(torch.bfloat16)
            v_pool = torch.randn((pool_blocks, Hkv, bs, hd), generator=gen, device="cuda").to(torch.bfloat16)
            perm = torch.from_numpy(synth.permutation(synth.SWEEP_SEED + ctx, pool_blocks).astype(np.int32)).cuda()
            tables = [perm[i * nblk:(i + 1) * nblk].contiguous() for i in range(n)]
            q = torch.randn(Hq * hd, generator=gen, device="cuda")
            o = torch.empty(Hq * hd, dtype=torch.float32, device="cuda")
            ws = torch.empty(max(mie.mie_paged_attn_workspace_bytes(Hq, Hkv, hd, ctx, bs), 256), dtype=torch.uint8,
                             device="cuda")
            stride = Hkv * bs * hd
            dt = graph_time(torch, [(lambda st, t=t: mie.mie_paged_attn_decode(
                q, k_pool, v_pool, stride, pool_blocks, t, ctx, Hq, Hkv, hd, bs, hd ** -0.5, o, ws, stream=st))
                for t in tables])
            out["attention"].append({"ctx": ctx, "us": dt * 1e6, "gbs": per_call / dt / 1e9,
                                     "frac": per_call / dt / 1e9 / peak, "launches": n})
            del k_pool, v_pool, tables
            torch.cuda.empty_cache()
        V = 128256
        if want("argmax"):
            n = max(least, int(total // (V * 4)) + 1)
            vs = [torch.randn(V, generator=gen, device="cuda") for _ in range(n)]
            am = torch.empty(1, dtype=torch.int32, device="cuda")
            wsa = torch.empty(mie.mie_argmax_workspace_bytes(V), dtype=torch.uint8, device="cuda")
            dt = graph_time(torch, [(lambda st, v=v: mie.mie_argmax(v, am, wsa, stream=st)) for v in vs])
            out["argmax"] = {"n": V, "us": dt * 1e6, "gbs": V * 4 / dt / 1e9, "launches": n}
            del vs
            torch.cuda.empty_cache()
    if clk:
        out["clocks"] = clk.summary()
    return out


def main():
    args = parse()
    if args.workload == "sweep":
        run_sweep(args)
        return
    if args.layers:
        from dataclasses import replace as _replace  # a truncated model for profiling captures
        synth_shape = _replace(synth.llama32_1b(args.fmt, args.head), n_layers=args.layers)
    else:
        synth_shape = None
    if args.workload == "prefill":
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        if args.gemm:
            import memory_bound_decode_dequant_gb300 as mie
            _, N, K = next(g for g in GEMM_SHAPES if g[0] == args.gemm)
            W = torch.randn(N, K, device="cuda").mul_(0.02).to(torch.bfloat16)
            planes = mie.mie_split_bf16(torch.randn(2048, K, device="cuda"))
            y = torch.empty(2048, N, device="cuda")
            for _ in range(max(1, args.steps)):
                mie.mie_gemm_bf16(W, planes, y)
            torch.cuda.synchronize()
            mie.mie_check()
            print(json.dumps({"gemm": args.gemm, "N": N, "K": K, "T": 2048, "launches": max(1, args.steps)}))
        else:
            print(json.dumps(prefill_measure(torch, measured_bf16_peak())), flush=True)
        return
    if args.workload == "slots":
        if args.impl == "reference":
            run_reference_slots(args)
        else:
            run_slots(args)
        return
    shape = synth_shape or synth.llama32_1b(args.fmt, args.head)
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
