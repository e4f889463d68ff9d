"""Python access to the oracle (mie_oracle.c) -- TEST INFRASTRUCTURE.

Only the tests, `__graft_entry__.smoke()` and the bench's CPU-baseline leg may import
this package.  It is a thin ctypes layer: every number it returns is computed by the
plain C code in mie_oracle.c (serial by default; set_threads(n) spreads independent
rows and heads over n host threads with bit-identical results).  It shares no code
with the CUDA library.

Parity pins: every function is pinned by a `-m "not gpu"` test.  The full-model logits
are "parity unpinned" beyond the composition of pinned parts (the pages print no
values for synthetic weights); the incremental-vs-no-cache invariant pins the cache
plumbing of the step.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, f"libmie_oracle.{platform.machine()}.so")
_lib = None

FMT = {"bf16": 0, "i8": 1, "q4_0": 2, "f32": 3, "q4_g64": 4, "q4_g128": 5}
# weights per f16 scale of the 4-bit formats
Q4_GROUP = {"q4_0": 32, "q4_g64": 64, "q4_g128": 128}
P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile mie_oracle.c with plain gcc; -ffp-contract=off keeps every multiply and
    add separately rounded, as the quantisers' rounding decisions require."""
    src = os.path.join(_HERE, "mie_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]
        try:  # OpenMP for the optional multi-threaded runs; without it the oracle is serial
            subprocess.check_call(base + ["-fopenmp", "-o", tmp, src, "-lm"], stderr=subprocess.DEVNULL)
        except subprocess.CalledProcessError:
            subprocess.check_call(base + ["-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("block_size", ctypes.c_int), ("act_bf16", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double)]


def lib():
    global _lib
    if _lib is not None:
        return _lib
    build()
    L = ctypes.CDLL(_SO)
    i, i64, f, d = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    sig = {
        "or_set_threads": (i, [i]),
        "or_max_threads": (i, []),
        "or_f32_to_bf16": (ctypes.c_uint16, [f]),
        "or_bf16_to_f32": (f, [ctypes.c_uint16]),
        "or_f32_to_f16": (ctypes.c_uint16, [f]),
        "or_f16_to_f32": (f, [ctypes.c_uint16]),
        "or_f32_to_bf16_n": (None, [P, i64, P]),
        "or_bf16_to_f32_n": (None, [P, i64, P]),
        "or_f32_to_f16_n": (None, [P, i64, P]),
        "or_f16_to_f32_n": (None, [P, i64, P]),
        "or_q4_0_quantize": (None, [P, i, i, P]),
        "or_q4_0_dequantize": (None, [P, i, i, P]),
        "or_q4_group": (i, [i]),
        "or_q4_quantize": (None, [P, i, i, i, P]),
        "or_q4_dequantize": (None, [P, i, i, i, P]),
        "or_i8_quantize": (None, [P, i, i, P, P]),
        "or_i8_dequantize": (None, [P, P, i, i, P]),
        "or_gemv": (None, [i, P, P, P, i, i, P]),
        "or_embed_row": (None, [i, P, P, i, i, i, P]),
        "or_rmsnorm": (None, [P, P, i, f, P]),
        "or_rope_table": (None, [i, i, d, P, P]),
        "or_rope_apply": (None, [P, i, i, P, P]),
        "or_swiglu": (None, [P, P, i, P]),
        "or_argmax": (i, [P, i]),
        "or_splitmix64": (ctypes.c_uint64, [ctypes.c_uint64, ctypes.c_uint64]),
        "or_sample_uniform": (d, [ctypes.c_uint64, i, i]),
        "or_sample": (i, [P, i, f, i, f, ctypes.c_uint64, i]),
        "or_attention_paged": (None, [P, P, P, i64, P, i, i, i, i, i, f, P]),
        "or_attention_contig": (None, [P, P, P, i, i, i, i, f, P]),
        "or_pool_create": (P, [i, i64]),
        "or_pool_destroy": (None, [P]),
        "or_pool_alloc": (i, [P]),
        "or_pool_incref": (i, [P, i]),
        "or_pool_decref": (i, [P, i]),
        "or_pool_refcount": (i, [P, i]),
        "or_pool_free_count": (i, [P]),
        "or_pool_data": (P, [P, i]),
        "or_table_writable": (i, [P, P, i, i]),
        "or_model_create": (P, [ctypes.POINTER(_Config), i, i]),
        "or_model_destroy": (None, [P]),
        "or_model_block_elems": (i64, [P]),
        "or_model_kv": (P, [P]),
        "or_model_set": (i, [P, i, i, i, P, P, i, i]),
        "or_decode_step": (i, [P, i, i, P, i, P]),
        "or_forward_nocache": (i, [P, P, i, P]),
        "or_decode_step_slots": (i, [P, i, P, P, P, i, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return a.ctypes.data if a is not None else None


# --------------------------------------------------------------------- conversions

def set_threads(n: int) -> int:
    """Host threads for the oracle's independent rows and heads (1 = serial); returns
    the count in effect (1 when built without OpenMP)."""
    return int(lib().or_set_threads(int(n)))


def max_threads() -> int:
    return int(lib().or_max_threads())


def to_bf16(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().or_f32_to_bf16_n(_p(x), x.size, _p(out))
    return out


def from_bf16(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().or_bf16_to_f32_n(_p(h), h.size, _p(out))
    return out


def to_f16(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().or_f32_to_f16_n(_p(x), x.size, _p(out))
    return out


def from_f16(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().or_f16_to_f32_n(_p(h), h.size, _p(out))
    return out


# --------------------------------------------------------------------- quantisers

def q4_0_quantize(w) -> np.ndarray:
    """fp32 [M, K] -> canonical Q4_0 bytes [M, ceil(K/32), 18]."""
    w = _c(w, np.float32)
    M, K = w.shape
    nb = (K + 31) // 32
    out = np.empty((M, nb, 18), np.uint8)
    lib().or_q4_0_quantize(_p(w), M, K, _p(out))
    return out


def q4_0_dequantize(wq, K: int) -> np.ndarray:
    wq = _c(wq, np.uint8)
    M = wq.shape[0]
    out = np.empty((M, K), np.float32)
    lib().or_q4_0_dequantize(_p(wq), M, K, _p(out))
    return out


def q4_quantize(w, group: int) -> np.ndarray:
    """fp32 [M, K] -> canonical 4-bit groups [M, ceil(K/group), 2 + group/2] bytes
    (group 32 is Q4_0)."""
    w = _c(w, np.float32)
    M, K = w.shape
    ng = (K + group - 1) // group
    out = np.empty((M, ng, 2 + group // 2), np.uint8)
    lib().or_q4_quantize(_p(w), M, K, group, _p(out))
    return out


def q4_dequantize(wq, K: int, group: int) -> np.ndarray:
    wq = _c(wq, np.uint8)
    M = wq.shape[0]
    out = np.empty((M, K), np.float32)
    lib().or_q4_dequantize(_p(wq), M, K, group, _p(out))
    return out


def i8_quantize(w):
    w = _c(w, np.float32)
    M, K = w.shape
    q = np.empty((M, K), np.int8)
    s = np.empty(M, np.float32)
    lib().or_i8_quantize(_p(w), M, K, _p(q), _p(s))
    return q, s


def i8_dequantize(q, s) -> np.ndarray:
    q = _c(q, np.int8)
    s = _c(s, np.float32)
    M, K = q.shape
    out = np.empty((M, K), np.float32)
    lib().or_i8_dequantize(_p(q), _p(s), M, K, _p(out))
    return out


class Mat:
    """A weight matrix in one canonical storage format, owned by Python."""

    def __init__(self, fmt: str, data: np.ndarray, rows: int, cols: int, scale=None):
        self.fmt, self.data, self.rows, self.cols, self.scale = fmt, data, rows, cols, scale

    @staticmethod
    def quantize(fmt: str, w) -> "Mat":
        w = _c(w, np.float32)
        M, K = w.shape
        if fmt == "bf16":
            return Mat(fmt, to_bf16(w), M, K)
        if fmt == "i8":
            q, s = i8_quantize(w)
            return Mat(fmt, q, M, K, s)
        if fmt in Q4_GROUP:
            return Mat(fmt, q4_quantize(w, Q4_GROUP[fmt]), M, K)
        if fmt == "f32":
            return Mat(fmt, w, M, K)
        raise ValueError(fmt)

    def dequantize(self) -> np.ndarray:
        if self.fmt == "bf16":
            return from_bf16(self.data).reshape(self.rows, self.cols)
        if self.fmt == "i8":
            return i8_dequantize(self.data, self.scale)
        if self.fmt in Q4_GROUP:
            return q4_dequantize(self.data, self.cols, Q4_GROUP[self.fmt])
        return self.data.reshape(self.rows, self.cols).copy()


# --------------------------------------------------------------------- ops

def gemv(mat: Mat, x) -> np.ndarray:
    x = _c(x, np.float32)
    assert x.size == mat.cols
    y = np.empty(mat.rows, np.float32)
    lib().or_gemv(FMT[mat.fmt], _p(mat.data), _p(mat.scale), _p(x), mat.rows, mat.cols, _p(y))
    return y


def embed_row(mat: Mat, token: int) -> np.ndarray:
    x = np.empty(mat.cols, np.float32)
    lib().or_embed_row(FMT[mat.fmt], _p(mat.data), _p(mat.scale), mat.rows, mat.cols, token, _p(x))
    return x


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x = _c(x, np.float32)
    g = _c(g, np.float32)
    out = np.empty_like(x)
    lib().or_rmsnorm(_p(x), _p(g), x.size, eps, _p(out))
    return out


def rope_table(n_pos: int, hd: int, base: float):
    c = np.empty((n_pos, hd // 2), np.float32)
    s = np.empty((n_pos, hd // 2), np.float32)
    lib().or_rope_table(n_pos, hd, base, _p(c), _p(s))
    return c, s


def rope_apply(v, n_heads: int, hd: int, cos_row, sin_row) -> np.ndarray:
    v = _c(v, np.float32).copy()
    cr = _c(cos_row, np.float32)
    sr = _c(sin_row, np.float32)
    lib().or_rope_apply(_p(v), n_heads, hd, _p(cr), _p(sr))
    return v


def swiglu(g, u) -> np.ndarray:
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    out = np.empty_like(g)
    lib().or_swiglu(_p(g), _p(u), g.size, _p(out))
    return out


def argmax(v) -> int:
    v = _c(v, np.float32)
    return int(lib().or_argmax(_p(v), v.size))


def attention_paged(q, k_pool, v_pool, block_stride: int, block_table, ctx: int, Hq: int,
                    Hkv: int, hd: int, bs: int, scale: float) -> np.ndarray:
    q = _c(q, np.float32)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    bt = _c(block_table, np.int32)
    out = np.empty(Hq * hd, np.float32)
    lib().or_attention_paged(_p(q), _p(k_pool), _p(v_pool), block_stride, _p(bt), ctx, Hq, Hkv,
                             hd, bs, scale, _p(out))
    return out


def attention_contig(q, k, v, ctx: int, Hq: int, Hkv: int, hd: int, scale: float) -> np.ndarray:
    q = _c(q, np.float32)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    out = np.empty(Hq * hd, np.float32)
    lib().or_attention_contig(_p(q), _p(k), _p(v), ctx, Hq, Hkv, hd, scale, _p(out))
    return out


# --------------------------------------------------------------------- sampling

def splitmix64(seed: int, i: int) -> int:
    return int(lib().or_splitmix64(seed & (2**64 - 1), i & (2**64 - 1)))


def sample_uniform(seed: int, pos: int, i: int) -> float:
    return float(lib().or_sample_uniform(seed & (2**64 - 1), pos, i))


def sample(logits, temperature: float, top_k: int = 0, top_p: float = 1.0, seed: int = 0, pos: int = 0) -> int:
    """Token drawn by temperature / top-k / top-p sampling (see or_sample)."""
    v = _c(logits, np.float32)
    return int(lib().or_sample(_p(v), v.size, temperature, top_k, top_p, seed & (2**64 - 1), pos))


# --------------------------------------------------------------------- block pool

class Pool:
    """The oracle's block pool (refcounts, LIFO free list, copy-on-write)."""

    def __init__(self, n_blocks: int, bytes_per_block: int):
        self.n_blocks, self.bytes_per_block = n_blocks, bytes_per_block
        self.h = lib().or_pool_create(n_blocks, bytes_per_block)

    def __del__(self):
        if getattr(self, "h", None):
            lib().or_pool_destroy(self.h)
            self.h = None

    def alloc(self) -> int:
        return lib().or_pool_alloc(self.h)

    def incref(self, i: int) -> int:
        return lib().or_pool_incref(self.h, i)

    def decref(self, i: int) -> int:
        return lib().or_pool_decref(self.h, i)

    def refcount(self, i: int) -> int:
        return lib().or_pool_refcount(self.h, i)

    def free_count(self) -> int:
        return lib().or_pool_free_count(self.h)

    def data(self, i: int) -> np.ndarray:
        ptr = lib().or_pool_data(self.h, i)
        buf = (ctypes.c_uint8 * self.bytes_per_block).from_address(ptr)
        return np.frombuffer(buf, dtype=np.uint8)

    def writable(self, table: np.ndarray, pos: int, block_size: int) -> int:
        assert table.dtype == np.int32 and table.flags.c_contiguous
        return lib().or_table_writable(self.h, table.ctypes.data, pos, block_size)


# --------------------------------------------------------------------- the model

class Model:
    """The oracle's decoder: canonical weights quantised by the oracle's own quantisers
    from the synth module's fp32 draws, a host KV pool, and the plain decode step."""

    def __init__(self, shape, n_kv_blocks: int, max_pos: int, weights: dict | None = None,
                 layers: int | None = None):
        self.shape = shape
        nl = shape.n_layers if layers is None else layers
        cfg = _Config(nl, shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                      shape.ffn, shape.vocab, shape.block_size, int(shape.act_bf16),
                      shape.rms_eps, shape.rope_theta)
        self.n_layers = nl
        self.h = lib().or_model_create(ctypes.byref(cfg), n_kv_blocks, max_pos)
        self.n_kv_blocks, self.max_pos = n_kv_blocks, max_pos
        self.block_elems = int(lib().or_model_block_elems(self.h))
        self._keep = []
        self.mats = {}
        ones_d = np.ones(shape.d_model, np.float32)
        self._keep.append(ones_d)
        which = {"qkv": 0, "o": 1, "gate": 2, "up": 3, "down": 4}
        for name, m, k in shape.tensors():
            if name.startswith("l") and int(name[1:].split(".")[0]) >= nl:
                continue
            w = weights[name] if weights and name in weights else None
            fmt = shape.head_fmt if name in ("head", "embed") else shape.wfmt
            if name == "embed":
                fmt = shape.wfmt
            mat = w if isinstance(w, Mat) else Mat.quantize(fmt, shape.weight(name) if w is None else w)
            self.mats[name] = mat
            if name == "head":
                self._set(100, 0, mat)
                if shape.tied:
                    self._set(101, 0, mat)
            elif name == "embed":
                self._set(101, 0, mat)
            else:
                layer, t = name[1:].split(".")
                self._set(which[t], int(layer), mat)
        for layer in range(nl):
            for t in (5, 6):
                lib().or_model_set(self.h, t, layer, FMT["f32"], _p(ones_d), None, 1, shape.d_model)
        lib().or_model_set(self.h, 102, 0, FMT["f32"], _p(ones_d), None, 1, shape.d_model)

    def _set(self, which, layer, mat: Mat):
        self._keep.append(mat)
        r = lib().or_model_set(self.h, which, layer, FMT[mat.fmt], _p(mat.data), _p(mat.scale),
                               mat.rows, mat.cols)
        assert r == 0

    def __del__(self):
        if getattr(self, "h", None):
            lib().or_model_destroy(self.h)
            self.h = None

    def kv(self) -> np.ndarray:
        """The KV pool as a live uint16 view: [n_blocks, n_layers, 2, Hkv, bs, hd]."""
        s = self.shape
        n = self.n_kv_blocks * self.block_elems
        buf = (ctypes.c_uint16 * n).from_address(lib().or_model_kv(self.h))
        return np.frombuffer(buf, dtype=np.uint16).reshape(
            self.n_kv_blocks, self.n_layers, 2, s.n_kv_heads, s.block_size, s.head_dim)

    def decode_step(self, token: int, pos: int, block_table) -> tuple[np.ndarray, int]:
        bt = _c(block_table, np.int32)
        logits = np.empty(self.shape.vocab, np.float32)
        r = lib().or_decode_step(self.h, int(token), int(pos), _p(bt), bt.size, _p(logits))
        if r < 0:
            raise ValueError("oracle decode step rejected its arguments")
        return logits, r

    def decode_step_slots(self, tokens, pos, block_tables) -> tuple[np.ndarray, np.ndarray]:
        """One step of every slot: tokens[s] at pos[s] through block_tables[s] (one row of
        the [n_slots, max_blocks] table per slot); returns ([n_slots, vocab] logits, argmax)."""
        t, p = _c(tokens, np.int32), _c(pos, np.int32)
        bt = _c(block_tables, np.int32)
        n = t.size
        assert p.size == n and bt.ndim == 2 and bt.shape[0] == n
        logits = np.empty((n, self.shape.vocab), np.float32)
        best = np.empty(n, np.int32)
        r = lib().or_decode_step_slots(self.h, n, _p(t), _p(p), _p(bt), bt.shape[1], _p(logits), _p(best))
        if r < 0:
            raise ValueError("oracle slot step rejected its arguments")
        return logits, best

    def forward_nocache(self, tokens) -> tuple[np.ndarray, int]:
        t = _c(tokens, np.int32)
        logits = np.empty(self.shape.vocab, np.float32)
        r = lib().or_forward_nocache(self.h, _p(t), t.size, _p(logits))
        if r < 0:
            raise ValueError("oracle forward rejected its arguments")
        return logits, r
