"""Seeded synthetic inputs for the decode-step workloads.

This module holds the workload recipes (model shapes, seeds, token streams) and the
random-number generators that both the oracle and the CUDA path draw their inputs
from.  It contains none of the decode step's arithmetic: no quantisation, no
bf16/f16 rounding, no matrix products.  Each side turns these fp32 arrays into its
own storage formats.

Shapes follow the pages' workloads:
  * "Writing an LLM inference engine from scratch in Rust", section "How a Llama
    model generates text": TinyLlama, 22 layers, d_model 2048, 32 query / 4 KV heads,
    SwiGLU 2048 -> 5632 -> 2048, vocabulary 32000.
  * "infer" (C++/CUDA engine for Llama-3.2-1B), per-kernel table: GEMV shapes
    3072x2048, 2048x2048, 16384x2048, 2048x8192, 128256x2048; 32 query / 8 KV heads.
Weights are N(0, 0.02), tokens uniform over the vocabulary; the "infer" page notes
that random weights with the real shapes suffice for tests and speed.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, f"libsynth.{platform.machine()}.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.<machine>.so next to it (gcc, no target-specific
    flags; one file per host architecture, so x86-64 and AArch64 builds sit side by side)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11",
                               "-ffp-contract=off", "-o", tmp, src, "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        lib.synth_u64.restype = ctypes.c_uint64
        lib.synth_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_normal_f32.restype = None
        lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_void_p,
                                         ctypes.c_int]
        lib.synth_uniform_i32.restype = None
        lib.synth_uniform_i32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
        lib.synth_permutation.restype = None
        lib.synth_permutation.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_void_p]
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def u64(seed: int, i: int) -> int:
    """Output i of the splitmix64 stream that starts at `seed`."""
    return int(_load().synth_u64(seed & (2**64 - 1), i))


def normal(seed: int, n: int, std: float = 1.0, mean: float = 0.0, offset: int = 0,
           out: np.ndarray | None = None) -> np.ndarray:
    """fp32 N(mean, std) elements offset .. offset+n-1 of the normal stream `seed`."""
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    if n:
        _load().synth_normal_f32(seed & (2**64 - 1), offset, n, float(mean), float(std),
                                 out.ctypes.data, _threads())
    return out


def uniform_int(seed: int, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    """int32 values uniform in [lo, hi)."""
    out = np.empty(n, dtype=np.int32)
    if n:
        _load().synth_uniform_i32(seed & (2**64 - 1), offset, n, lo, hi, out.ctypes.data)
    return out


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1 (int32)."""
    out = np.empty(max(n, 0), dtype=np.int32)
    if n:
        _load().synth_permutation(seed & (2**64 - 1), n, out.ctypes.data)
    return out


# --------------------------------------------------------------------------- workloads

@dataclass(frozen=True)
class ModelShape:
    """One Llama-style decoder shape plus its storage formats.

    wfmt / head_fmt are "bf16", "i8" (one fp32 scale per row), "q4_0" (blocks of 32
    four-bit values with one f16 scale) or "q4_g64" / "q4_g128" (groups of 64 / 128
    four-bit values with one f16 scale).  act_bf16 rounds each GEMV input vector to
    bf16 (the TinyLlama workload's "bf16 activations"); the residual stream stays fp32.
    """
    name: str
    index: int               # position in the workload list; part of every seed
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    tied: bool
    rope_theta: float
    rms_eps: float = 1e-5
    wfmt: str = "bf16"
    head_fmt: str = "bf16"
    act_bf16: bool = False
    block_size: int = 16
    weight_std: float = 0.02

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    def tensors(self):
        """(name, rows, cols) of every weight matrix, in seed order: for each layer
        qkv, o, gate, up, down; then the LM head; then the embedding when untied."""
        out = []
        d, f = self.d_model, self.ffn
        for layer in range(self.n_layers):
            out += [(f"l{layer}.qkv", self.qkv_rows, d),
                    (f"l{layer}.o", d, self.n_heads * self.head_dim),
                    (f"l{layer}.gate", f, d),
                    (f"l{layer}.up", f, d),
                    (f"l{layer}.down", d, f)]
        out.append(("head", self.vocab, d))
        if not self.tied:
            out.append(("embed", self.vocab, d))
        return out

    def seed(self, name: str) -> int:
        names = [t[0] for t in self.tensors()]
        return 0x4D4945 + 1000 * self.index + names.index(name)

    def shape(self, name: str):
        for t in self.tensors():
            if t[0] == name:
                return t[1], t[2]
        raise KeyError(name)

    def weight(self, name: str, rows: slice | None = None) -> np.ndarray:
        """fp32 weights of tensor `name` ([rows, cols]); `rows` draws only a slice."""
        m, k = self.shape(name)
        r0, r1 = (0, m) if rows is None else (rows.start or 0, m if rows.stop is None else rows.stop)
        w = normal(self.seed(name), (r1 - r0) * k, std=self.weight_std, offset=r0 * k)
        return w.reshape(r1 - r0, k)

    def tokens(self, n: int, stream: int = 0) -> np.ndarray:
        return uniform_int(0x544F4B + self.index + 7919 * stream, n, 0, self.vocab)

    def weight_bytes(self, fmt: str | None = None) -> int:
        """Bytes one decode step streams for all GEMV weights (embedding gather excluded)."""
        total = 0
        for name, m, k in self.tensors():
            if name == "embed":
                continue
            f = self.head_fmt if name == "head" else (fmt or self.wfmt)
            total += matrix_bytes(f, m, k)
        return total

    def kv_bytes_per_token(self) -> int:
        """bf16 K and V of one position, every layer."""
        return self.n_layers * 2 * self.n_kv_heads * self.head_dim * 2

    def decode_bytes(self, first_pos: int, n_steps: int) -> float:
        """Mean algorithmic bytes of one step over n_steps consecutive decode steps whose
        first writes position first_pos: the weights once, plus the K/V of every position
        the step attends to (p + 1 of them at position p)."""
        mean_ctx = first_pos + (n_steps + 1) / 2
        return self.weight_bytes() + self.kv_bytes_per_token() * mean_ctx


# weights per f16 scale of the 4-bit formats
Q4_GROUP = {"q4_0": 32, "q4_g64": 64, "q4_g128": 128}


def matrix_bytes(fmt: str, m: int, k: int) -> int:
    """Algorithmic bytes of an m x k matrix in a storage format (unpadded)."""
    if fmt == "bf16":
        return m * k * 2
    if fmt == "i8":
        return m * k + 4 * m
    if fmt in Q4_GROUP:  # one f16 scale and group/2 bytes of 4-bit codes per group
        g = Q4_GROUP[fmt]
        return m * ((k + g - 1) // g) * (2 + g // 2)
    if fmt == "f32":
        return m * k * 4
    raise ValueError(fmt)


def gemv_bytes(fmt: str, m: int, k: int) -> int:
    """Algorithmic bytes of one y = W x launch: the weights once, an fp32 x in, an fp32
    y out."""
    return matrix_bytes(fmt, m, k) + 4 * k + 4 * m


TINY = ModelShape("tiny", 0, n_layers=2, d_model=256, n_heads=8, n_kv_heads=2, head_dim=32,
                  ffn=688, vocab=1024, tied=False, rope_theta=10000.0,
                  wfmt="q4_0", head_fmt="q4_0")
TINYLLAMA = ModelShape("tinyllama-1.1b", 1, n_layers=22, d_model=2048, n_heads=32,
                       n_kv_heads=4, head_dim=64, ffn=5632, vocab=32000, tied=False,
                       rope_theta=10000.0, wfmt="q4_0", head_fmt="q4_0", act_bf16=True)
LLAMA32_1B = ModelShape("llama-3.2-1b", 2, n_layers=16, d_model=2048, n_heads=32,
                        n_kv_heads=8, head_dim=64, ffn=8192, vocab=128256, tied=True,
                        rope_theta=500000.0, wfmt="bf16", head_fmt="bf16")


def llama32_1b(fmt: str, head: str | None = None) -> ModelShape:
    """The Llama-3.2-1B shape in one of its storage variants: "bf16", "i8" (per-row
    scale), or a 4-bit format ("q4_0", "q4_g64", "q4_g128") for the layers with the
    tied head/embedding in int8 unless `head` names another format (e.g. the same
    4-bit format: the all-int4 variants)."""
    if head is None:
        head = {"bf16": "bf16", "i8": "i8"}.get(fmt, "i8")
    return replace(LLAMA32_1B, wfmt=fmt, head_fmt=head)


# Per-kernel sweep at the Llama-3.2-1B decode shapes.
SWEEP_GEMV = [("qkv", 3072, 2048), ("o", 2048, 2048), ("gate_up", 16384, 2048),
              ("down", 2048, 8192), ("lm_head", 128256, 2048)]
SWEEP_ATTN_CTX = [512, 2048, 8192]
SWEEP_SEED = 0x535745


@dataclass
class SlotWorkload:
    """Continuous-batching step: slot contexts, shared prefix, retire/admit cadence."""
    n_slots: int = 8
    ctx_lo: int = 128
    ctx_hi: int = 4096
    shared_slots: int = 4
    shared_prefix: int = 512
    steps: int = 256
    admit_every: int = 32
    admit_len: int = 256
    seed: int = 0x534C54
    ctx: np.ndarray = field(default=None)

    def __post_init__(self):
        if self.ctx is None:
            c = uniform_int(self.seed, self.n_slots, self.ctx_lo, self.ctx_hi + 1)
            c[: self.shared_slots] = np.maximum(c[: self.shared_slots], self.shared_prefix)
            self.ctx = c
