"""ctypes binding of libmie.so; names follow the C ABI in include/mie.h."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmie.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "mie.h")

Q4_GROUP = {"q4_0": 32, "q4_g64": 64, "q4_g128": 128}  # weights per f16 scale
FMT = {"bf16": 0, "i8": 1, "q4_0": 2, "f32": 3, "q4_g64": 4, "q4_g128": 5}
STATUS = {0: "MIE_OK", 1: "MIE_E_ARG", 2: "MIE_E_SHAPE", 3: "MIE_E_OOM", 4: "MIE_E_CUDA",
          5: "MIE_E_TIMEOUT", 6: "MIE_E_STATE", 7: "MIE_E_DEVICE"}

__all__ = ["lib", "MieError", "FMT", "LIB_PATH", "exported_names", "header_functions",
           "mie_convert_bf16", "mie_quantize_i8", "mie_quantize_q4_0", "mie_q4_0_pack",
           "mie_q4_0_packed_bytes", "mie_gemv_bf16", "mie_gemv_i8", "mie_gemv_q4_0",
           "mie_quantize_q4", "mie_q4_packed_bytes", "mie_q4_pack", "mie_gemv_q4", "Q4_GROUP",
           "mie_paged_attn_decode", "mie_paged_attn_workspace_bytes", "mie_paged_attn_decode_noalloc",
           "mie_argmax", "mie_split_bf16", "mie_gemm_bf16", "mie_paged_attn_prefill",
           "mie_argmax_workspace_bytes", "mie_check", "mie_hbm_read_probe", "mie_sample", "mie_sample_workspace_bytes", "Pool", "Config", "Model",
           "DeviceArray"]


class MieError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


P = ctypes.c_void_p
I, I64, F, SZ = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


class Config(ctypes.Structure):
    """mie_config."""
    _fields_ = [("n_layers", I), ("d_model", I), ("n_heads", I), ("n_kv_heads", I),
                ("head_dim", I), ("ffn", I), ("vocab", I), ("tied", I), ("block_size", I),
                ("act_bf16", I), ("rms_eps", F), ("rope_theta", F), ("wfmt", I), ("head_fmt", I),
                ("embed_fmt", I), ("n_kv_blocks", I), ("max_slots", I), ("max_pos", I)]


_SIGS = {
    "mie_last_error": (ctypes.c_char_p, []),
    "mie_status_string": (ctypes.c_char_p, [I]),
    "mie_convert_bf16": (I, [P, I64, P, P]),
    "mie_quantize_i8": (I, [P, I, I, P, P, P]),
    "mie_quantize_q4_0": (I, [P, I, I, P, P]),
    "mie_q4_0_packed_bytes": (SZ, [I, I]),
    "mie_q4_0_pack": (I, [P, I, I, P, P]),
    "mie_quantize_q4": (I, [P, I, I, I, P, P]),
    "mie_q4_packed_bytes": (SZ, [I, I, I]),
    "mie_q4_pack": (I, [P, I, I, I, P, P]),
    "mie_gemv_bf16": (I, [P, P, P, I, I, P]),
    "mie_gemv_i8": (I, [P, P, P, P, I, I, P]),
    "mie_gemv_q4_0": (I, [P, P, P, I, I, P]),
    "mie_gemv_q4": (I, [P, I, P, P, I, I, P]),
    "mie_split_bf16": (I, [P, I64, P, P, P, P]),
    "mie_gemm_bf16": (I, [P, I, I, P, P, P, I, P, I64, I, P]),
    "mie_paged_attn_prefill": (I, [P, P, P, I64, I, P, I, I, I, I, I, I, I, F, P, P]),
    "mie_prefill": (I, [P, P, I, ctypes.c_int32, P, I]),
    "mie_paged_attn_workspace_bytes": (SZ, [I, I, I, I, I]),
    "mie_paged_attn_decode": (I, [P, P, P, I64, I, P, I, I, I, I, I, I, F, P, P, SZ, P]),
    "mie_paged_attn_decode_noalloc": (I, [P, P, P, I64, I, P, I, I, I, I, I, I, F, P, P]),
    "mie_argmax_workspace_bytes": (SZ, [I]),
    "mie_argmax": (I, [P, I, P, P, SZ, P]),
    "mie_check": (I, [P]),
    "mie_hbm_read_probe": (I, [P, SZ, P, I, I, P]),
    "mie_sample_workspace_bytes": (SZ, []),
    "mie_sample": (I, [P, I, F, I, F, ctypes.c_uint64, ctypes.c_int32, P, P, SZ, P]),
    "mie_set_sampling": (I, [P, F, I, F, ctypes.c_uint64]),
    "mie_pool_create": (I, [I, ctypes.POINTER(P)]),
    "mie_pool_destroy": (None, [P]),
    "mie_pool_alloc": (I, [P, ctypes.POINTER(ctypes.c_int32)]),
    "mie_pool_incref": (I, [P, ctypes.c_int32]),
    "mie_pool_decref": (I, [P, ctypes.c_int32]),
    "mie_pool_refcount": (I, [P, ctypes.c_int32]),
    "mie_pool_free_count": (I, [P]),
    "mie_pool_writable": (I, [P, P, I, I, ctypes.POINTER(ctypes.c_int32),
                              ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "mie_create": (I, [ctypes.POINTER(Config), P, ctypes.POINTER(P)]),
    "mie_destroy": (None, [P]),
    "mie_load_weights": (I, [P, ctypes.c_char_p, I, P, SZ, ctypes.POINTER(ctypes.c_int64), I, P]),
    "mie_ctx_pool": (P, [P]),
    "mie_kv_pool": (P, [P]),
    "mie_kv_block_elems": (I64, [P]),
    "mie_kv_copy_block": (I, [P, ctypes.c_int32, ctypes.c_int32]),
    "mie_kv_writable": (I, [P, P, I, ctypes.POINTER(ctypes.c_int32)]),
    "mie_decode_step": (I, [P, ctypes.c_int32, ctypes.c_int32, P, I, P, P]),
    "mie_decode_step_sync": (I, [P, ctypes.c_int32, ctypes.c_int32, P, I, P, P]),
    "mie_decode_continue": (I, [P, I]),
    "mie_decode_step_slots": (I, [P, I, P, P, P, I, P, P]),
    "mie_sync": (I, [P]),
    "mie_step_launches": (I, [P]),
    "mie_set_step_mode": (I, [P, I]),
    "mie_step_mode": (I, [P]),
    "mie_slot_step_launches": (I, [P]),
    "mie_set_trace": (I, [P, P, SZ, ctypes.POINTER(I), ctypes.POINTER(I)]),
    "mie_debug_stall": (I, [P, I, ctypes.c_long]),
    "mie_verify_step": (I, [P, P, I, ctypes.c_int32, P, I, P, P]),
    "mie_lookup_propose": (I, [P, I, I, I, I, P]),
    "mie_spec_gate_bytes": (SZ, []),
    "mie_spec_gate_init": (None, [P, I, F, I, I]),
    "mie_spec_gate_open": (I, [P]),
    "mie_spec_gate_record": (None, [P, I, I]),
    "mie_generate": (I, [P, P, I, I, P, I, I, P]),
}

_lib = None


def lib():
    """The loaded libmie.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Every function name that include/mie.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mie_[a-z0-9_]+)\s*\(", text)))


def exported_names() -> list[str]:
    return [n for n in header_functions() if hasattr(lib(), n)]


def _check(status: int, what: str = ""):
    if status != 0:
        msg = lib().mie_last_error().decode(errors="replace")
        raise MieError(status, f"{what}: {msg}" if what else msg)


# --------------------------------------------------------------------- torch glue

def _torch():
    import torch
    return torch


def _dev(t, dtype=None, name="tensor"):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def mie_convert_bf16(w, out=None, stream=None):
    torch = _torch()
    out = torch.empty(w.shape, dtype=torch.bfloat16, device=w.device) if out is None else out
    _check(lib().mie_convert_bf16(_dev(w, torch.float32, "w"), w.numel(), _dev(out, torch.bfloat16, "out"),
                                  _stream(stream)), "mie_convert_bf16")
    return out


def mie_quantize_i8(w, stream=None):
    torch = _torch()
    M, K = w.shape
    q = torch.empty((M, K), dtype=torch.int8, device=w.device)
    s = torch.empty((M,), dtype=torch.float32, device=w.device)
    _check(lib().mie_quantize_i8(_dev(w, torch.float32, "w"), M, K, q.data_ptr(), s.data_ptr(), _stream(stream)),
           "mie_quantize_i8")
    return q, s


def mie_quantize_q4_0(w, stream=None):
    torch = _torch()
    M, K = w.shape
    out = torch.empty((M, (K + 31) // 32, 18), dtype=torch.uint8, device=w.device)
    _check(lib().mie_quantize_q4_0(_dev(w, torch.float32, "w"), M, K, out.data_ptr(), _stream(stream)),
           "mie_quantize_q4_0")
    return out


def mie_q4_0_packed_bytes(M: int, K: int) -> int:
    return int(lib().mie_q4_0_packed_bytes(M, K))


def mie_q4_0_pack(blocks, M: int, K: int, stream=None):
    torch = _torch()
    out = torch.empty(mie_q4_0_packed_bytes(M, K), dtype=torch.uint8, device=blocks.device)
    _check(lib().mie_q4_0_pack(_dev(blocks, torch.uint8, "blocks"), M, K, out.data_ptr(), _stream(stream)),
           "mie_q4_0_pack")
    return out


def mie_quantize_q4(w, group: int, stream=None):
    """fp32 [M, K] device tensor -> canonical 4-bit groups [M, ceil(K/group), 2 + group/2]."""
    torch = _torch()
    M, K = w.shape
    out = torch.empty((M, (K + group - 1) // group, 2 + group // 2), dtype=torch.uint8, device=w.device)
    _check(lib().mie_quantize_q4(_dev(w, torch.float32, "w"), M, K, group, out.data_ptr(), _stream(stream)),
           "mie_quantize_q4")
    return out


def mie_q4_packed_bytes(M: int, K: int, group: int) -> int:
    return int(lib().mie_q4_packed_bytes(M, K, group))


def mie_q4_pack(groups, M: int, K: int, group: int, stream=None):
    torch = _torch()
    out = torch.empty(mie_q4_packed_bytes(M, K, group), dtype=torch.uint8, device=groups.device)
    _check(lib().mie_q4_pack(_dev(groups, torch.uint8, "groups"), M, K, group, out.data_ptr(), _stream(stream)),
           "mie_q4_pack")
    return out


def mie_gemv_q4(packed, group: int, x, M: int, K: int, y=None, stream=None):
    torch = _torch()
    y = _y(y, M, packed.device)
    _check(lib().mie_gemv_q4(_dev(packed, torch.uint8, "packed"), group, _dev(x, torch.float32, "x"),
                             _dev(y, torch.float32, "y"), M, K, _stream(stream)), "mie_gemv_q4")
    return y


def _y(y, M, device):
    torch = _torch()
    return torch.empty(M, dtype=torch.float32, device=device) if y is None else y


def mie_gemv_bf16(W, x, y=None, stream=None):
    torch = _torch()
    M, K = W.shape
    y = _y(y, M, W.device)
    _check(lib().mie_gemv_bf16(_dev(W, torch.bfloat16, "W"), _dev(x, torch.float32, "x"),
                               _dev(y, torch.float32, "y"), M, K, _stream(stream)), "mie_gemv_bf16")
    return y


def mie_gemv_i8(W, scale, x, y=None, stream=None):
    torch = _torch()
    M, K = W.shape
    y = _y(y, M, W.device)
    _check(lib().mie_gemv_i8(_dev(W, torch.int8, "W"), _dev(scale, torch.float32, "scale"),
                             _dev(x, torch.float32, "x"), _dev(y, torch.float32, "y"), M, K, _stream(stream)),
           "mie_gemv_i8")
    return y


def mie_gemv_q4_0(packed, x, M: int, K: int, y=None, stream=None):
    torch = _torch()
    y = _y(y, M, packed.device)
    _check(lib().mie_gemv_q4_0(_dev(packed, torch.uint8, "packed"), _dev(x, torch.float32, "x"),
                               _dev(y, torch.float32, "y"), M, K, _stream(stream)), "mie_gemv_q4_0")
    return y


def mie_split_bf16(x, planes: int = 3, stream=None):
    """x (fp32, any shape) -> list of `planes` (1 to 3) bf16 planes hi, mid, lo of x."""
    torch = _torch()
    out = [torch.empty(x.shape, dtype=torch.bfloat16, device=x.device) for _ in range(planes)]
    ptr = [_dev(p, torch.bfloat16, "plane") for p in out] + [None] * (3 - planes)
    _check(lib().mie_split_bf16(_dev(x, torch.float32, "x"), x.numel(), ptr[0], ptr[1], ptr[2], _stream(stream)),
           "mie_split_bf16")
    return out


def mie_gemm_bf16(W, planes, y=None, accumulate: bool = False, stream=None):
    """y[t][n] (+)= sum_k W[n][k] (sum of the planes)[t][k] on the tensor cores; W [N][K],
    planes: 1 to 3 bf16 [T][K] tensors (hi, mid, lo); y [T][ldy >= N] fp32."""
    torch = _torch()
    N, K = W.shape
    T = planes[0].shape[0]
    if y is None:
        y = torch.empty((T, N), dtype=torch.float32, device=W.device)
    ptr = [_dev(p, torch.bfloat16, "plane") for p in planes] + [None] * (3 - len(planes))
    _check(lib().mie_gemm_bf16(_dev(W, torch.bfloat16, "W"), N, K, ptr[0], ptr[1], ptr[2], T,
                               _dev(y, torch.float32, "y"), y.stride(0), int(bool(accumulate)), _stream(stream)),
           "mie_gemm_bf16")
    return y


def mie_paged_attn_prefill(q, k_pool, v_pool, block_stride: int, n_pool_blocks: int, block_table,
                           pos0: int, Hq: int, Hkv: int, hd: int, bs: int, scale: float, out=None, stream=None):
    """Causal attention of the T = q.shape[0] positions pos0 .. pos0+T-1; q [T][Hq*hd] fp32."""
    torch = _torch()
    T = q.shape[0]
    if out is None:
        out = torch.empty((T, Hq * hd), dtype=torch.float32, device=q.device)
    _check(lib().mie_paged_attn_prefill(
        _dev(q, torch.float32, "q"), _dev(k_pool, None, "k_pool"), _dev(v_pool, None, "v_pool"), block_stride,
        n_pool_blocks, _dev(block_table, torch.int32, "block_table"), block_table.numel(), pos0, T, Hq, Hkv, hd, bs,
        scale, _dev(out, torch.float32, "out"), _stream(stream)), "mie_paged_attn_prefill")
    return out


def mie_paged_attn_workspace_bytes(Hq, Hkv, hd, ctx_len, bs) -> int:
    return int(lib().mie_paged_attn_workspace_bytes(Hq, Hkv, hd, ctx_len, bs))


def mie_paged_attn_decode(q, k_pool, v_pool, block_stride: int, n_pool_blocks: int, block_table,
                          ctx_len: int, Hq: int, Hkv: int, hd: int, bs: int, scale: float,
                          out=None, workspace=None, stream=None):
    torch = _torch()
    if out is None:
        out = torch.empty(Hq * hd, dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = max(mie_paged_attn_workspace_bytes(Hq, Hkv, hd, ctx_len, bs), 256)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(lib().mie_paged_attn_decode(
        _dev(q, torch.float32, "q"), _dev(k_pool, None, "k_pool"), _dev(v_pool, None, "v_pool"),
        block_stride, n_pool_blocks, _dev(block_table, torch.int32, "block_table"), block_table.numel(),
        ctx_len, Hq, Hkv, hd, bs, scale, _dev(out, torch.float32, "out"), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)), "mie_paged_attn_decode")
    return out


def mie_paged_attn_decode_noalloc(q, k_pool, v_pool, block_stride: int, n_pool_blocks: int, block_table,
                                  ctx_len: int, Hq: int, Hkv: int, hd: int, bs: int, scale: float,
                                  out=None, stream=None):
    """mie_paged_attn_decode without a workspace: for callers that cannot allocate
    device memory; its scratch is the library's built-in 1 MiB array (see mie.h)."""
    torch = _torch()
    if out is None:
        out = torch.empty(Hq * hd, dtype=torch.float32, device=q.device)
    _check(lib().mie_paged_attn_decode_noalloc(
        _dev(q, torch.float32, "q"), _dev(k_pool, None, "k_pool"), _dev(v_pool, None, "v_pool"),
        block_stride, n_pool_blocks, _dev(block_table, torch.int32, "block_table"), block_table.numel(),
        ctx_len, Hq, Hkv, hd, bs, scale, _dev(out, torch.float32, "out"), _stream(stream)),
        "mie_paged_attn_decode_noalloc")
    return out


def mie_argmax_workspace_bytes(n: int) -> int:
    return int(lib().mie_argmax_workspace_bytes(n))


def mie_argmax(v, out=None, workspace=None, stream=None):
    torch = _torch()
    if out is None:
        out = torch.empty(1, dtype=torch.int32, device=v.device)
    if workspace is None:
        workspace = torch.empty(mie_argmax_workspace_bytes(v.numel()), dtype=torch.uint8, device=v.device)
    _check(lib().mie_argmax(_dev(v, torch.float32, "v"), v.numel(), _dev(out, torch.int32, "out"),
                            workspace.data_ptr(), workspace.numel(), _stream(stream)), "mie_argmax")
    return out


def mie_hbm_read_probe(buf, xor_out=None, load_bytes: int = 32, blocks_per_sm: int = 2, stream=None):
    """Reads every byte of the device tensor `buf` once; returns the int32 device tensor
    that receives the XOR of its 32-bit words."""
    torch = _torch()
    if xor_out is None:
        xor_out = torch.empty(1, dtype=torch.int32, device=buf.device)
    _check(lib().mie_hbm_read_probe(_dev(buf, None, "buf"), buf.numel() * buf.element_size(),
                                    _dev(xor_out, torch.int32, "xor_out"), load_bytes, blocks_per_sm,
                                    _stream(stream)), "mie_hbm_read_probe")
    return xor_out


def mie_sample_workspace_bytes() -> int:
    return int(lib().mie_sample_workspace_bytes())


def mie_sample(logits, temperature: float, top_k: int = 0, top_p: float = 1.0, seed: int = 0, pos: int = 0,
               out=None, workspace=None, stream=None):
    """The token drawn from the device logits tensor (int32 device tensor, returned)."""
    torch = _torch()
    if out is None:
        out = torch.empty(1, dtype=torch.int32, device=logits.device)
    if workspace is None:
        workspace = torch.empty(mie_sample_workspace_bytes(), dtype=torch.uint8, device=logits.device)
    _check(lib().mie_sample(_dev(logits, torch.float32, "logits"), logits.numel(), float(temperature), int(top_k),
                            float(top_p), seed & (2**64 - 1), int(pos), _dev(out, torch.int32, "out"),
                            workspace.data_ptr(), workspace.numel(), _stream(stream)), "mie_sample")
    return out


def mie_check(stream=None):
    _check(lib().mie_check(_stream(stream)), "mie_check")


# --------------------------------------------------------------------- block pool

class Pool:
    """mie_pool: refcounted KV block ids with a LIFO free list (host only)."""

    def __init__(self, n_blocks: int = 0, handle=None):
        self._own = handle is None
        if handle is None:
            h = P()
            _check(lib().mie_pool_create(n_blocks, ctypes.byref(h)), "mie_pool_create")
            handle = h.value
        self.h = handle

    def __del__(self):
        if getattr(self, "_own", False) and getattr(self, "h", None):
            lib().mie_pool_destroy(self.h)
            self.h = None

    def alloc(self) -> int:
        i = ctypes.c_int32(-1)
        st = lib().mie_pool_alloc(self.h, ctypes.byref(i))
        if st not in (0, 3):
            _check(st, "mie_pool_alloc")
        return i.value

    def incref(self, i: int) -> int:
        return lib().mie_pool_incref(self.h, i)

    def decref(self, i: int) -> int:
        return lib().mie_pool_decref(self.h, i)

    def refcount(self, i: int) -> int:
        return lib().mie_pool_refcount(self.h, i)

    def free_count(self) -> int:
        return lib().mie_pool_free_count(self.h)

    def writable(self, table: np.ndarray, pos: int, block_size: int):
        """(status, block, copy_src, copy_dst); the table is updated in place.  After a
        split (copy_src >= 0) the sequence still holds copy_src: queue the copy, then
        decref(copy_src)."""
        assert table.dtype == np.int32 and table.flags.c_contiguous
        b, s, d = ctypes.c_int32(-1), ctypes.c_int32(-1), ctypes.c_int32(-1)
        st = lib().mie_pool_writable(self.h, table.ctypes.data, pos, block_size, ctypes.byref(b),
                                     ctypes.byref(s), ctypes.byref(d))
        return st, b.value, s.value, d.value


# --------------------------------------------------------------------- model

class DeviceArray:
    """A device buffer owned by the library, exposed to torch via __cuda_array_interface__."""

    def __init__(self, ptr: int, shape, typestr: str, owner):
        self._owner = owner
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


class Model:
    """mie_ctx: weights in GPU layouts, the paged KV pool and the graph-captured step."""

    def __init__(self, cfg: dict, stream=None):
        c = Config(**cfg)
        self.cfg = dict(cfg)
        h = P()
        _check(lib().mie_create(ctypes.byref(c), _stream(stream) if stream is not None else None, ctypes.byref(h)),
               "mie_create")
        self.h = h.value
        self.pool = Pool(handle=lib().mie_ctx_pool(self.h))

    def close(self):
        if getattr(self, "h", None):
            lib().mie_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()

    def load_weights(self, name: str, data: np.ndarray, fmt: str = "f32", scale: np.ndarray | None = None,
                     cols: int | None = None):
        """Copies host data (numpy) into the context: fp32 [rows, cols] (quantised on the
        GPU), or the tensor's own format in canonical layout."""
        data = np.ascontiguousarray(data)
        if data.ndim == 1:
            shape = (data.shape[0],)
        elif fmt == "q4_0":
            shape = (data.shape[0], cols)
        else:
            shape = data.shape[:2]
        arr = (ctypes.c_int64 * len(shape))(*shape)
        sc = None
        if scale is not None:
            scale = np.ascontiguousarray(scale, dtype=np.float32)
            sc = scale.ctypes.data
        _check(lib().mie_load_weights(self.h, name.encode(), FMT[fmt], data.ctypes.data, data.nbytes, arr,
                                      len(shape), sc), f"mie_load_weights({name})")

    @property
    def block_elems(self) -> int:
        return int(lib().mie_kv_block_elems(self.h))

    def kv(self):
        """The device KV pool as a torch uint16-bits tensor
        [n_kv_blocks, n_layers, 2, n_kv_heads, block_size, head_dim] (bf16 bit patterns)."""
        torch = _torch()
        c = self.cfg
        shape = (c["n_kv_blocks"], c["n_layers"], 2, c["n_kv_heads"], c["block_size"], c["head_dim"])
        arr = DeviceArray(lib().mie_kv_pool(self.h), shape, "<i2", self)
        return torch.as_tensor(arr, device="cuda")

    def kv_copy_block(self, src: int, dst: int):
        _check(lib().mie_kv_copy_block(self.h, src, dst), "mie_kv_copy_block")

    def kv_writable(self, table: np.ndarray, pos: int) -> int:
        """Copy-on-write on the context's pool (split, copy queued, old reference
        dropped); the host table is updated in place; returns the block to write."""
        assert table.dtype == np.int32 and table.flags.c_contiguous
        b = ctypes.c_int32(-1)
        _check(lib().mie_kv_writable(self.h, table.ctypes.data, int(pos), ctypes.byref(b)), "mie_kv_writable")
        return b.value

    def decode_step(self, token: int, pos: int, block_table, logits_out=None, argmax_out=None):
        torch = _torch()
        _check(lib().mie_decode_step(self.h, int(token), int(pos), _dev(block_table, torch.int32, "block_table"),
                                     block_table.numel(),
                                     None if logits_out is None else _dev(logits_out, torch.float32, "logits"),
                                     None if argmax_out is None else _dev(argmax_out, torch.int32, "argmax")),
               "mie_decode_step")

    def decode_step_sync(self, token: int, pos: int, block_table, logits_out=None) -> int:
        """One step with host token / position in and the next token read back (waits)."""
        torch = _torch()
        nxt = ctypes.c_int32(0)
        _check(lib().mie_decode_step_sync(self.h, int(token), int(pos), _dev(block_table, torch.int32, "block_table"),
                                          block_table.numel(),
                                          None if logits_out is None else _dev(logits_out, torch.float32, "logits"),
                                          ctypes.byref(nxt)),
               "mie_decode_step_sync")
        return int(nxt.value)

    def decode_continue(self, n_steps: int):
        _check(lib().mie_decode_continue(self.h, n_steps), "mie_decode_continue")

    def decode_step_slots(self, tokens, pos, block_tables, logits_out=None, argmax_out=None):
        torch = _torch()
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        p = np.ascontiguousarray(pos, dtype=np.int32)
        n_slots, max_blocks = block_tables.shape
        _check(lib().mie_decode_step_slots(self.h, n_slots, t.ctypes.data, p.ctypes.data,
                                           _dev(block_tables, torch.int32, "block_tables"), max_blocks,
                                           None if logits_out is None else _dev(logits_out, torch.float32, "logits"),
                                           None if argmax_out is None else _dev(argmax_out, torch.int32, "argmax")),
               "mie_decode_step_slots")

    def sync(self):
        _check(lib().mie_sync(self.h), "mie_sync")

    @property
    def launches(self) -> int:
        return int(lib().mie_step_launches(self.h))

    @property
    def slot_launches(self) -> int:
        return int(lib().mie_slot_step_launches(self.h))

    PERSISTENT, CHAIN = 0, 1

    def set_step_mode(self, mode: int):
        _check(lib().mie_set_step_mode(self.h, mode), "mie_set_step_mode")

    @property
    def step_mode(self) -> int:
        return int(lib().mie_step_mode(self.h))

    def verify_step(self, tokens, pos: int, block_table, logits_out=None, argmax_out=None):
        """Positions pos .. pos+n-1 of one sequence (host tokens) as n slots sharing one
        block table (device int32 [max_blocks])."""
        torch = _torch()
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(lib().mie_verify_step(self.h, t.ctypes.data, t.size, int(pos),
                                     _dev(block_table, torch.int32, "block_table"), block_table.numel(),
                                     None if logits_out is None else _dev(logits_out, torch.float32, "logits"),
                                     None if argmax_out is None else _dev(argmax_out, torch.int32, "argmax")),
               "mie_verify_step")

    def prefill(self, tokens, pos0: int, block_table):
        """K/V of the host tokens at positions pos0 .. pos0+n-1 into the cache, on the
        tensor cores (no logits: the next decode step gives them)."""
        torch = _torch()
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(lib().mie_prefill(self.h, t.ctypes.data, t.size, int(pos0),
                                 _dev(block_table, torch.int32, "block_table"), block_table.numel()),
               "mie_prefill")

    def generate(self, prompt, n_new: int, block_table, spec_max: int = 1):
        """Greedy generation (prompt through mie_prefill, then few-slot passes, speculative
        for spec_max > 1); returns (generated tokens, {passes, proposed, accepted})."""
        torch = _torch()
        ids = np.zeros(len(prompt) + n_new, np.int32)
        ids[: len(prompt)] = prompt
        stats = (ctypes.c_int * 3)()
        _check(lib().mie_generate(self.h, ids.ctypes.data, len(prompt), n_new,
                                  _dev(block_table, torch.int32, "block_table"), block_table.numel(), spec_max, stats),
               "mie_generate")
        return ids[len(prompt):].copy(), {"passes": stats[0], "proposed": stats[1], "accepted": stats[2]}

    def set_sampling(self, temperature: float, top_k: int = 0, top_p: float = 1.0, seed: int = 0):
        _check(lib().mie_set_sampling(self.h, float(temperature), int(top_k), float(top_p), seed & (2**64 - 1)),
               "mie_set_sampling")

    def debug_stall(self, phase: int, wait_polls: int = 0):
        """Testing aid: phase `phase` of the persistent step waits for an input nobody
        writes, and every wait gives up after wait_polls rounds (phase < 0 restores)."""
        _check(lib().mie_debug_stall(self.h, int(phase), int(wait_polls)), "mie_debug_stall")

    STAGE_TRACE, STAGE_POINTS = 1024, 4

    def set_trace(self, enable: bool = True, stages: bool = False):
        """Records the persistent step's timeline into a device tensor
        [n_phases, n_ctas, 5] of int64 nanoseconds (returned), or switches it off.  With
        stages=True the tensor also carries the per-stage stamps and points inside each
        phase (instrumented build), and (phases, stages, points) views of it are
        returned: stages [n_ctas, 1024, 4], points [n_phases, n_ctas, 8]."""
        torch = _torch()
        npz, nct = I(0), I(0)
        if not enable:
            _check(lib().mie_set_trace(self.h, None, 0, ctypes.byref(npz), ctypes.byref(nct)), "mie_set_trace")
            self._trace = None
            return None
        _check(lib().mie_set_trace(self.h, None, 0, ctypes.byref(npz), ctypes.byref(nct)), "mie_set_trace")
        n_ph = npz.value * nct.value * 5
        n_st = nct.value * self.STAGE_TRACE * self.STAGE_POINTS if stages else 0
        n_sub = npz.value * nct.value * 8 if stages else 0
        flat = torch.zeros(n_ph + n_st + n_sub, dtype=torch.int64, device="cuda")
        _check(lib().mie_set_trace(self.h, flat.data_ptr(), flat.numel() * 8, None, None), "mie_set_trace")
        self._trace = flat
        ph = flat[:n_ph].view(npz.value, nct.value, 5)
        if not stages:
            return ph
        return (ph, flat[n_ph:n_ph + n_st].view(nct.value, self.STAGE_TRACE, self.STAGE_POINTS),
                flat[n_ph + n_st:].view(npz.value, nct.value, 8))


# ------------------------------------------------ the context and pool calls by C name
#
# The same entry points as the methods above, under the names include/mie.h gives them:
# `ctx` is a Model (mie_ctx), `pool` a Pool (mie_pool).

def mie_last_error() -> str:
    return lib().mie_last_error().decode(errors="replace")


def mie_status_string(status: int) -> str:
    return lib().mie_status_string(int(status)).decode(errors="replace")


def mie_pool_create(n_blocks: int) -> Pool:
    return Pool(n_blocks)


def mie_pool_destroy(pool: Pool) -> None:
    if pool._own and pool.h:
        lib().mie_pool_destroy(pool.h)
        pool.h = None


def mie_pool_alloc(pool: Pool) -> int:
    """A block id, or -1 when the pool is exhausted."""
    return pool.alloc()


def mie_pool_incref(pool: Pool, block: int) -> None:
    _check(pool.incref(block), "mie_pool_incref")


def mie_pool_decref(pool: Pool, block: int) -> None:
    _check(pool.decref(block), "mie_pool_decref")


def mie_pool_refcount(pool: Pool, block: int) -> int:
    return pool.refcount(block)


def mie_pool_free_count(pool: Pool) -> int:
    return pool.free_count()


def mie_pool_writable(pool: Pool, table: np.ndarray, pos: int, block_size: int):
    """(block, copy_src, copy_dst) with the table updated in place; MieError (out of
    memory) when no block is free.  After a split the caller still holds copy_src and
    drops it with mie_pool_decref once the copy is queued."""
    st, b, s, d = pool.writable(table, pos, block_size)
    _check(st, "mie_pool_writable")
    return b, s, d


def mie_create(cfg: dict, stream=None) -> Model:
    return Model(cfg, stream)


def mie_destroy(ctx: Model) -> None:
    ctx.close()


def mie_load_weights(ctx: Model, name: str, data: np.ndarray, fmt: str = "f32",
                     scale: np.ndarray | None = None, cols: int | None = None) -> None:
    ctx.load_weights(name, data, fmt, scale, cols)


def mie_ctx_pool(ctx: Model) -> Pool:
    return ctx.pool


def mie_kv_pool(ctx: Model):
    return ctx.kv()


def mie_kv_block_elems(ctx: Model) -> int:
    return ctx.block_elems


def mie_kv_copy_block(ctx: Model, src: int, dst: int) -> None:
    ctx.kv_copy_block(src, dst)


def mie_kv_writable(ctx: Model, table: np.ndarray, pos: int) -> int:
    return ctx.kv_writable(table, pos)


def mie_decode_step(ctx: Model, token: int, pos: int, block_table, logits_out=None, argmax_out=None) -> None:
    ctx.decode_step(token, pos, block_table, logits_out, argmax_out)


def mie_decode_step_sync(ctx: Model, token: int, pos: int, block_table, logits_out=None) -> int:
    return ctx.decode_step_sync(token, pos, block_table, logits_out)


def mie_decode_continue(ctx: Model, n_steps: int) -> None:
    ctx.decode_continue(n_steps)


def mie_decode_step_slots(ctx: Model, tokens, pos, block_tables, logits_out=None, argmax_out=None) -> None:
    ctx.decode_step_slots(tokens, pos, block_tables, logits_out, argmax_out)


def mie_set_step_mode(ctx: Model, mode: int) -> None:
    ctx.set_step_mode(mode)


def mie_step_mode(ctx: Model) -> int:
    return ctx.step_mode


def mie_set_trace(ctx: Model, enable: bool = True):
    return ctx.set_trace(enable)


def mie_sync(ctx: Model) -> None:
    ctx.sync()


def mie_set_sampling(ctx: Model, temperature: float, top_k: int = 0, top_p: float = 1.0, seed: int = 0) -> None:
    ctx.set_sampling(temperature, top_k, top_p, seed)


def mie_verify_step(ctx: Model, tokens, pos: int, block_table, logits_out=None, argmax_out=None) -> None:
    ctx.verify_step(tokens, pos, block_table, logits_out, argmax_out)


def mie_prefill(ctx: Model, tokens, pos0: int, block_table) -> None:
    ctx.prefill(tokens, pos0, block_table)


def mie_generate(ctx: Model, prompt, n_new: int, block_table, spec_max: int = 1):
    return ctx.generate(prompt, n_new, block_table, spec_max)


def mie_lookup_propose(ids, min_ngram: int, max_ngram: int, k: int) -> list:
    """Prompt-lookup guesses for the context ids (host)."""
    a = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.zeros(max(k, 1), np.int32)
    n = lib().mie_lookup_propose(a.ctypes.data, a.size, min_ngram, max_ngram, k, out.ctypes.data)
    return [int(v) for v in out[:n]]


class SpecGate:
    """mie_spec_gate: the acceptance gate of speculative decoding (host)."""

    def __init__(self, window: int = 10, threshold: float = 0.3, pause: int = 5, pause_max: int = 80):
        self._buf = ctypes.create_string_buffer(int(lib().mie_spec_gate_bytes()))
        lib().mie_spec_gate_init(self._buf, window, threshold, pause, pause_max)

    def open(self) -> bool:
        return bool(lib().mie_spec_gate_open(self._buf))

    def record(self, proposed: int, accepted: int) -> None:
        lib().mie_spec_gate_record(self._buf, proposed, accepted)


def mie_spec_gate_bytes() -> int:
    return int(lib().mie_spec_gate_bytes())


def mie_spec_gate_init(gate: SpecGate, window: int, threshold: float, pause: int, pause_max: int) -> None:
    lib().mie_spec_gate_init(gate._buf, window, threshold, pause, pause_max)


def mie_spec_gate_open(gate: SpecGate) -> bool:
    return gate.open()


def mie_spec_gate_record(gate: SpecGate, proposed: int, accepted: int) -> None:
    gate.record(proposed, accepted)


def mie_debug_stall(ctx: Model, phase: int, wait_polls: int = 0) -> None:
    ctx.debug_stall(phase, wait_polls)


def mie_step_launches(ctx: Model) -> int:
    return ctx.launches


def mie_slot_step_launches(ctx: Model) -> int:
    return ctx.slot_launches


__all__ += ["mie_last_error", "mie_status_string", "mie_pool_create", "mie_pool_destroy", "mie_pool_alloc",
            "mie_pool_incref", "mie_pool_decref", "mie_pool_refcount", "mie_pool_free_count",
            "mie_pool_writable", "mie_create", "mie_destroy", "mie_load_weights", "mie_ctx_pool",
            "mie_kv_pool", "mie_kv_block_elems", "mie_kv_copy_block", "mie_kv_writable", "mie_decode_step",
            "mie_decode_step_sync", "mie_decode_continue", "mie_decode_step_slots", "mie_set_step_mode", "mie_step_mode",
            "mie_set_trace", "mie_set_sampling", "mie_debug_stall", "mie_sync", "mie_verify_step", "mie_prefill", "mie_generate",
            "mie_lookup_propose", "SpecGate", "mie_spec_gate_bytes", "mie_spec_gate_init", "mie_spec_gate_open",
            "mie_spec_gate_record", "mie_step_launches", "mie_slot_step_launches"]
