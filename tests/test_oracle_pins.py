"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test checks an oracle function against something other than itself: IEEE
conversions from numpy/torch, closed forms, invariants, special cases that reduce to a
library routine (numpy matmul, scipy softmax/expit), or brute force on tiny inputs.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import synth

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------- conversions

def test_f16_roundtrip_all_patterns(orc):
    """f16 -> f32 equals numpy's IEEE binary16 decode for every bit pattern."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.from_f16(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_matches_numpy_rne(orc):
    """fp32 -> f16 rounding (nearest even, subnormals, overflow) equals numpy's."""
    vals = [0.0, -0.0, 1.0, 65504.0, 65519.0, 65520.0, 1e6, 2.0**-24, 2.0**-25, 3 * 2.0**-26,
            2.0**-14, 2.0**-14 - 2.0**-25, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, np.inf, -np.inf]
    x = np.concatenate([np.array(vals, np.float32),
                        RNG.standard_normal(200000).astype(np.float32) * 0.01,
                        (RNG.standard_normal(100000) * 1e-5).astype(np.float32),
                        (RNG.standard_normal(100000) * 3e4).astype(np.float32),
                        # exact halfway points between neighbouring f16 values
                        ((np.arange(1, 2048, dtype=np.float32) + 0.5) * 2.0**-10).astype(np.float32)])
    ours = orc.to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f32_to_bf16_matches_torch_rne(orc):
    """fp32 -> bf16 rounding equals torch's round-to-nearest-even conversion."""
    torch = pytest.importorskip("torch")
    x = np.concatenate([RNG.standard_normal(300000).astype(np.float32),
                        (RNG.standard_normal(1000) * 1e-39).astype(np.float32),
                        np.array([0.0, -0.0, 3.389e38, 3.4e38, np.inf, -np.inf, 1.0 + 2.0**-8,
                                  1.0 + 3 * 2.0**-8, 1.0 + 2.0**-8 + 2.0**-20], np.float32)])
    # exact ties: low 16 bits 0x8000
    ties = (RNG.integers(0x3F000000, 0x40000000, 5000, dtype=np.uint32) & 0xFFFF0000) | 0x8000
    x = np.concatenate([x, ties.view(np.float32)])
    ours = orc.to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = orc.from_bf16(ours)
    assert np.array_equal(back.view(np.uint32), ours.astype(np.uint32) << 16)


# ----------------------------------------------------------------- Q4_0

def _blocks(q):
    """Split canonical blocks into (scale bits, 32 codes)."""
    h = q[..., 0].astype(np.uint16) | (q[..., 1].astype(np.uint16) << 8)
    qs = q[..., 2:]
    codes = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)
    return h, codes


def test_q4_0_idempotent(orc):
    """quantize(dequantize(quantize(w))) == quantize(w) byte for byte."""
    w = synth.normal(11, 64 * 256, std=0.02).reshape(64, 256)
    q1 = orc.q4_0_quantize(w)
    q2 = orc.q4_0_quantize(orc.q4_0_dequantize(q1, 256))
    assert np.array_equal(q1, q2)


def test_q4_0_max_element_codes_to_zero(orc):
    """The largest-magnitude element maps exactly to -8: code 0, value -8h."""
    w = synth.normal(12, 128 * 64, std=0.02).reshape(128, 64)
    q = orc.q4_0_quantize(w)
    h, codes = _blocks(q)
    wb = w.reshape(128, 2, 32)
    idx = np.abs(wb).argmax(axis=-1)
    assert np.all(np.take_along_axis(codes, idx[..., None], -1) == 0)
    deq = orc.q4_0_dequantize(q, 64).reshape(128, 2, 32)
    hv = h.view(np.float16).astype(np.float32)
    assert np.array_equal(np.take_along_axis(deq, idx[..., None], -1)[..., 0], -8 * hv)
    # the stored scale is the f16 rounding of m / -8
    m = np.take_along_axis(wb, idx[..., None], -1)[..., 0]
    assert np.array_equal(h, (m / -8).astype(np.float16).view(np.uint16))


def test_q4_0_all_codes_roundtrip_and_nibble_order(orc):
    """A hand-built block holding every code 0..15 round-trips exactly, and byte j
    carries element j (low nibble) and element j+16 (high nibble)."""
    hv = np.float32(np.float16(0.00390625))  # 2^-8: exact in f16
    codes = np.array([0, 5, 1, 15, 2, 14, 3, 13, 4, 12, 6, 11, 7, 10, 9, 8] * 2, np.int64)
    codes[16:] = codes[16:][::-1]
    w = (hv * (codes - 8)).astype(np.float32)[None, :]
    q = orc.q4_0_quantize(w)
    h, got = _blocks(q)
    assert h[0, 0] == np.float16(hv).view(np.uint16)
    assert np.array_equal(got[0, 0], codes)
    assert np.array_equal(q[0, 0, 2:], (codes[:16] | (codes[16:] << 4)).astype(np.uint8))
    assert np.array_equal(orc.q4_0_dequantize(q, 32), w)


def test_q4_0_zero_block_and_ragged_tail(orc):
    """A zero block stores d = +0 / -8 = -0 and code 8 everywhere; a ragged row is
    zero-padded so the padding codes to 8 (exactly 0) and the real elements are
    unchanged."""
    q = orc.q4_0_quantize(np.zeros((1, 32), np.float32))
    h, codes = _blocks(q)
    assert h[0, 0] == 0x8000 and np.all(codes == 8)
    assert np.all(orc.q4_0_dequantize(q, 32) == 0)
    w = synth.normal(13, 3 * 40, std=0.02).reshape(3, 40)
    q = orc.q4_0_quantize(w)
    assert q.shape == (3, 2, 18)
    _, codes = _blocks(q)
    assert np.all(codes[:, 1, 8:] == 8)
    wp = np.zeros((3, 64), np.float32)
    wp[:, :40] = w
    assert np.array_equal(orc.q4_0_quantize(wp), q)


def test_q4_0_error_bound(orc):
    """Round-to-nearest on the grid h*(q-8), q in 0..15: |w - w'| <= |h|/2 except
    where the code saturates at 15 (the side opposite the max element can only reach
    7|h|), plus the max element's own f16 rounding of d."""
    w = synth.normal(14, 256 * 128, std=0.02).reshape(256, 128)
    q = orc.q4_0_quantize(w)
    deq = orc.q4_0_dequantize(q, 128)
    h, codes = _blocks(q)
    hv = np.abs(h.view(np.float16).astype(np.float64))[..., None]
    wb = np.abs(w.astype(np.float64)).reshape(256, 4, 32)
    err = np.abs(w.astype(np.float64) - deq).reshape(256, 4, 32)
    edge = hv * 8 * 2.0**-10  # 8 |d - h|, |d - h| <= |h| 2^-11 (f16 rounding)
    bound = np.maximum(hv * 0.5, np.where(codes == 15, wb - 7 * hv, 0)) + edge + 1e-12
    assert np.all(err <= bound)
    assert np.all(deq.reshape(256, 4, 32) >= -8 * hv - 1e-12)


def test_q4_0_bias_identity():
    """[RUST] Lesson 6: sum((w+8) x) - 8 sum(x) = sum(w x), exact over the rationals."""
    xs = [Fraction(float(v)) for v in synth.normal(15, 32)]
    n = [int(v) for v in synth.uniform_int(16, 32, 0, 16)]
    lhs = sum(Fraction(ni - 8) * xi for ni, xi in zip(n, xs))
    rhs = sum(Fraction(ni) * xi for ni, xi in zip(n, xs)) - 8 * sum(xs)
    assert lhs == rhs


# ----------------------------------------------------------------- 4-bit groups of 64 / 128

def _groups(q, GS):
    """(scale bits [M, ng], codes [M, ng, GS]) of canonical 4-bit groups: each group is
    its f16 scale then GS/32 sub-blocks of 16 bytes in the Q4_0 nibble order."""
    h = q[..., 0].astype(np.uint16) | (q[..., 1].astype(np.uint16) << 8)
    sub = q[..., 2:].reshape(q.shape[0], q.shape[1], GS // 32, 16)
    codes = np.concatenate([sub & 0x0F, sub >> 4], axis=-1).reshape(q.shape[0], q.shape[1], GS)
    return h, codes


@pytest.mark.parametrize("shape", [(1, 1), (3, 40), (4, 256), (5, 688), (2, 2048)])
def test_q4_group_32_is_q4_0(orc, shape):
    """Groups of 32 are Q4_0 byte for byte, ragged rows included."""
    M, K = shape
    w = synth.normal(40 + K, M * K, std=0.02).reshape(M, K)
    assert np.array_equal(orc.q4_quantize(w, 32), orc.q4_0_quantize(w))
    assert np.array_equal(orc.q4_dequantize(orc.q4_quantize(w, 32), K, 32),
                          orc.q4_0_dequantize(orc.q4_0_quantize(w), K))


@pytest.mark.parametrize("GS", [64, 128])
def test_q4_group_one_scale_per_group(orc, GS):
    """One f16 scale per group of GS: the group's largest-magnitude element codes to 0
    (value -8h), the stored scale is f16(m / -8), every element of the group dequantises
    to h * (code - 8) with that one scale, and quantising the dequantised matrix gives
    the same bytes (idempotence)."""
    M, K = 96, 512
    w = synth.normal(41 + GS, M * K, std=0.02).reshape(M, K)
    q = orc.q4_quantize(w, GS)
    assert q.shape == (M, K // GS, 2 + GS // 2)
    h, codes = _groups(q, GS)
    wg = w.reshape(M, K // GS, GS)
    idx = np.abs(wg).argmax(axis=-1)
    assert np.all(np.take_along_axis(codes, idx[..., None], -1) == 0)
    m = np.take_along_axis(wg, idx[..., None], -1)[..., 0]
    assert np.array_equal(h, (m / -8).astype(np.float16).view(np.uint16))
    hv = h.view(np.float16).astype(np.float32)
    deq = orc.q4_dequantize(q, K, GS).reshape(M, K // GS, GS)
    assert np.array_equal(deq, hv[..., None] * (codes.astype(np.float32) - 8))
    assert np.array_equal(orc.q4_quantize(deq.reshape(M, K), GS), q)


def test_q4_group_layout_hand_built(orc):
    """A hand-built group of 128 with every code in every sub-block round-trips, and its
    bytes are the scale then four 16-byte sub-blocks, byte j of sub-block b holding code
    32b + j (low nibble) and code 32b + j + 16 (high nibble)."""
    hv = np.float32(np.float16(0.0078125))  # 2^-7: exact in f16
    base = np.array([0, 5, 1, 15, 2, 14, 3, 13, 4, 12, 6, 11, 7, 10, 9, 8], np.int64)
    codes = np.concatenate([np.roll(base, b) if b % 2 == 0 else np.roll(base[::-1], b) for b in range(8)])
    codes[0] = 0  # the group's extreme (-8h) comes first and is unique
    codes[1:][codes[1:] == 0] = 1
    w = (hv * (codes - 8)).astype(np.float32)[None, :]
    q = orc.q4_quantize(w, 128)
    assert q.shape == (1, 1, 66)
    assert (int(q[0, 0, 0]) | (int(q[0, 0, 1]) << 8)) == int(np.float16(hv).view(np.uint16))
    for b in range(4):
        sub = codes[32 * b:32 * b + 32]
        assert np.array_equal(q[0, 0, 2 + 16 * b:18 + 16 * b], (sub[:16] | (sub[16:] << 4)).astype(np.uint8))
    assert np.array_equal(orc.q4_dequantize(q, 128, 128), w)


@pytest.mark.parametrize("GS", [64, 128])
def test_q4_group_ragged_tail_and_error_bound(orc, GS):
    """A row whose length is not a multiple of GS is zero-padded (pads code to 8, the
    real elements as if the zeros were there); every element lies within half a step of
    its group's grid, up to the saturated top code and the f16 rounding of the scale."""
    M, K = 7, 688
    w = synth.normal(43 + GS, M * K, std=0.02).reshape(M, K)
    q = orc.q4_quantize(w, GS)
    ng = (K + GS - 1) // GS
    assert q.shape == (M, ng, 2 + GS // 2)
    h, codes = _groups(q, GS)
    assert np.all(codes.reshape(M, ng * GS)[:, K:] == 8)
    wp = np.zeros((M, ng * GS), np.float32)
    wp[:, :K] = w
    assert np.array_equal(orc.q4_quantize(wp, GS), q)
    deq = orc.q4_dequantize(q, K, GS)
    hv = np.abs(h.view(np.float16).astype(np.float64))
    hv_el = np.repeat(hv, GS, axis=1)[:, :K]
    c_el = codes.reshape(M, ng * GS)[:, :K]
    wa = np.abs(w.astype(np.float64))
    err = np.abs(w.astype(np.float64) - deq)
    bound = np.maximum(hv_el * 0.5, np.where(c_el == 15, wa - 7 * hv_el, 0)) + hv_el * 8 * 2.0**-10 + 1e-12
    assert np.all(err <= bound)


@pytest.mark.parametrize("fmt", ["q4_g64", "q4_g128"])
def test_q4_group_embedding_row_is_the_dequantised_row(orc, fmt):
    """The embedding gather from a 4-bit table returns exactly the dequantised row."""
    w = synth.normal(45, 9 * 300, std=0.02).reshape(9, 300)
    mat = orc.Mat.quantize(fmt, w)
    deq = mat.dequantize()
    for t in (0, 4, 8):
        assert np.array_equal(orc.embed_row(mat, t), deq[t])


# ----------------------------------------------------------------- int8

def test_i8_quantizer(orc):
    w = synth.normal(21, 64 * 300, std=0.02).reshape(64, 300)
    w[3] = 0.0
    q, s = orc.i8_quantize(w)
    assert s[3] == 0 and np.all(q[3] == 0)
    live = np.arange(64) != 3
    amax = np.abs(w).max(axis=1)
    assert np.array_equal(s[live], (amax / np.float32(127))[live].astype(np.float32))
    idx = np.abs(w).argmax(axis=1)
    assert np.all(np.abs(q[live, idx[live]]) == 127)
    assert np.all(np.sign(q[live, idx[live]]) == np.sign(w[live, idx[live]]))
    deq = orc.i8_dequantize(q, s)
    assert np.all(np.abs(deq - w) <= s[:, None] * 0.5 * (1 + 1e-5) + 1e-12)
    q2, s2 = orc.i8_quantize(deq)
    assert np.array_equal(q2, q)


# ----------------------------------------------------------------- GEMV

@pytest.mark.parametrize("fmt", ["bf16", "i8", "q4_0", "q4_g64", "q4_g128", "f32"])
@pytest.mark.parametrize("shape", [(1, 1), (1, 32), (7, 40), (33, 688), (5, 2048), (64, 31)])
def test_gemv_brute_force(orc, fmt, shape):
    """The oracle GEMV equals the fp64 matrix-vector product of the dequantised
    weights (numpy) rounded to fp32, within the fp64 summation error."""
    M, K = shape
    w = synth.normal(31 + M, M * K, std=0.02).reshape(M, K)
    x = synth.normal(32 + K, K)
    mat = orc.Mat.quantize(fmt, w)
    y = orc.gemv(mat, x)
    if fmt == "i8":  # the dequantised weight s*q is exact in fp64
        wd = mat.scale.astype(np.float64)[:, None] * mat.data.astype(np.float64)
    else:
        wd = mat.dequantize().astype(np.float64)
    ref = wd @ x.astype(np.float64)
    mag = np.abs(wd) @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(y - ref) <= np.abs(ref) * 2.0**-24 + mag * K * 2.0**-52 + 1e-30)


def test_gemv_is_not_transposed(orc):
    """A matrix with one non-zero entry picks exactly one input into one output."""
    w = np.zeros((5, 9), np.float32)
    w[3, 7] = 2.0
    x = np.arange(9, dtype=np.float32)
    for fmt in ("bf16", "i8", "q4_0"):
        y = orc.gemv(orc.Mat.quantize(fmt, w), x)
        assert np.array_equal(y, np.array([0, 0, 0, 14, 0], np.float32)), fmt


# ----------------------------------------------------------------- RMSNorm, RoPE, SwiGLU, argmax

def test_rmsnorm_invariants(orc):
    x = synth.normal(41, 2048) * 3
    g = np.ones(2048, np.float32)
    y = orc.rmsnorm(x, g, 1e-5)
    ms = np.mean(x.astype(np.float64) ** 2)
    assert abs(np.mean(y.astype(np.float64) ** 2) - ms / (ms + 1e-5)) < 1e-6
    # scale invariance (eps negligible at this scale)
    y2 = orc.rmsnorm(x * 64, g, 1e-5)
    assert np.allclose(y2, y, rtol=2e-6, atol=0)
    # the gain multiplies elementwise
    gg = synth.normal(42, 2048)
    assert np.allclose(orc.rmsnorm(x, gg, 1e-5), y * gg, rtol=3e-7, atol=1e-30)
    # eps dominates a tiny vector: y = x / sqrt(eps)
    t = np.full(8, 1e-6, np.float32)
    assert np.allclose(orc.rmsnorm(t, np.ones(8, np.float32), 1e-5), t / np.sqrt(1e-5 + 1e-12), rtol=1e-6)


def test_rope_table_closed_forms(orc):
    c, s = orc.rope_table(64, 64, 10000.0)
    assert np.all(c[0] == 1) and np.all(s[0] == 0)
    # pair 0 rotates by exactly pos radians
    p = np.arange(64)
    assert np.array_equal(c[:, 0], np.cos(p.astype(np.float64)).astype(np.float32))
    assert np.array_equal(s[:, 0], np.sin(p.astype(np.float64)).astype(np.float32))
    # pair i at position 1 rotates by base^(-2i/hd): the frequencies form a geometric series
    ang = np.arctan2(s[1].astype(np.float64), c[1].astype(np.float64))
    ratios = ang[1:] / ang[:-1]
    assert np.allclose(ratios, 10000.0 ** (-2 / 64), rtol=1e-5)


def test_rope_is_rotate_half_rotation(orc):
    hd, H = 64, 4
    c, s = orc.rope_table(300, hd, 500000.0)
    v = synth.normal(51, H * hd)
    assert np.array_equal(orc.rope_apply(v, H, hd, c[0], s[0]), v)
    r = orc.rope_apply(v, H, hd, c[123], s[123]).reshape(H, hd).astype(np.float64)
    v2 = v.reshape(H, hd).astype(np.float64)
    n0 = v2[:, :32] ** 2 + v2[:, 32:] ** 2
    n1 = r[:, :32] ** 2 + r[:, 32:] ** 2
    assert np.allclose(n0, n1, rtol=1e-6)
    # single pair (hd = 2): a textbook 2-D rotation by pos radians
    c2, s2 = orc.rope_table(10, 2, 10000.0)
    a = np.array([0.3, -1.7], np.float32)
    th = 7.0
    rot = np.array([[math.cos(th), -math.sin(th)], [math.sin(th), math.cos(th)]])
    assert np.allclose(orc.rope_apply(a, 1, 2, c2[7], s2[7]), rot @ a.astype(np.float64), rtol=1e-6)


def test_rope_relative_position(orc):
    """<R(m) q, R(n) k> depends only on m - n."""
    hd = 64
    c, s = orc.rope_table(2100, hd, 10000.0)
    q = synth.normal(52, hd)
    k = synth.normal(53, hd)
    dots = []
    for m, n in [(5, 0), (105, 100), (2005, 2000)]:
        qr = orc.rope_apply(q, 1, hd, c[m], s[m]).astype(np.float64)
        kr = orc.rope_apply(k, 1, hd, c[n], s[n]).astype(np.float64)
        dots.append(qr @ kr)
    assert np.allclose(dots, dots[0], rtol=2e-5, atol=1e-5)
    # composition: R(a) R(b) = R(a + b)
    ab = orc.rope_apply(orc.rope_apply(q, 1, hd, c[300], s[300]), 1, hd, c[400], s[400])
    assert np.allclose(ab, orc.rope_apply(q, 1, hd, c[700], s[700]), atol=2e-5)


def test_swiglu(orc):
    g = np.concatenate([[0.0, 50.0, -50.0, -1000.0], synth.normal(61, 1000) * 4]).astype(np.float32)
    u = synth.normal(62, g.size) + 1
    a = orc.swiglu(g, u)
    assert a[0] == 0 and a[3] == 0
    assert np.isclose(a[1], 50.0 * u[1], rtol=1e-7)
    ref = (g.astype(np.float64) * scipy.special.expit(g.astype(np.float64)) * u).astype(np.float32)
    assert np.allclose(a, ref, rtol=2.0**-23, atol=1e-30)


def test_argmax_first_max(orc):
    v = synth.normal(71, 128256)
    assert orc.argmax(v) == int(np.argmax(v))
    v[[17, 99, 100000]] = v.max() + 1
    assert orc.argmax(v) == 17
    assert orc.argmax(np.full(5, -np.inf, np.float32)) == 0


# ----------------------------------------------------------------- attention

def _kv(seed, ctx, Hkv, hd):
    k = (synth.normal(seed, ctx * Hkv * hd)).reshape(ctx, Hkv, hd)
    v = (synth.normal(seed + 1, ctx * Hkv * hd)).reshape(ctx, Hkv, hd)
    return k, v


def test_attention_brute_force(orc):
    """Against scipy's softmax and an fp64 product, query head h reading KV head h/group."""
    import oracle
    Hq, Hkv, hd, ctx = 8, 2, 32, 37
    k, v = _kv(81, ctx, Hkv, hd)
    kb, vb = oracle.to_bf16(k), oracle.to_bf16(v)
    kf, vf = oracle.from_bf16(kb).astype(np.float64), oracle.from_bf16(vb).astype(np.float64)
    q = synth.normal(83, Hq * hd)
    scale = np.float32(1 / math.sqrt(hd))
    out = orc.attention_contig(q, kb, vb, ctx, Hq, Hkv, hd, scale).reshape(Hq, hd)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        p = scipy.special.softmax(kf[:, g, :] @ q[h * hd:(h + 1) * hd].astype(np.float64) * float(scale))
        assert np.allclose(out[h], p @ vf[:, g, :], rtol=1e-6, atol=1e-7)


def test_attention_special_cases(orc):
    import oracle
    Hq, Hkv, hd = 8, 2, 32
    k, v = _kv(84, 20, Hkv, hd)
    kb, vb = oracle.to_bf16(k), oracle.to_bf16(v)
    q = synth.normal(85, Hq * hd)
    # ctx 1: the output is v_0 exactly
    out = orc.attention_contig(q, kb, vb, 1, Hq, Hkv, hd, 0.17).reshape(Hq, hd)
    vf = oracle.from_bf16(vb).reshape(20, Hkv, hd)
    for h in range(Hq):
        assert np.array_equal(out[h], vf[0, h // 4])
    # empty context: zeros
    assert np.all(orc.attention_contig(q, kb, vb, 0, Hq, Hkv, hd, 0.17) == 0)
    # GQA equals MHA with each KV head repeated for its query heads
    kr = np.repeat(kb.reshape(20, Hkv, hd), 4, axis=1)
    vr = np.repeat(vb.reshape(20, Hkv, hd), 4, axis=1)
    a = orc.attention_contig(q, kb, vb, 20, Hq, Hkv, hd, 0.17)
    b = orc.attention_contig(q, kr, vr, 20, Hq, Hq, hd, 0.17)
    assert np.array_equal(a, b)


def test_paged_equals_contiguous(orc):
    """A random permutation of physical blocks read in logical order gives the same bits."""
    import oracle
    Hq, Hkv, hd, bs, ctx = 32, 8, 64, 16, 200
    nblk = (ctx + bs - 1) // bs
    k, v = _kv(86, nblk * bs, Hkv, hd)
    kb, vb = oracle.to_bf16(k), oracle.to_bf16(v)
    q = synth.normal(88, Hq * hd)
    perm = synth.permutation(89, 40)[:nblk]
    # pool: [40 blocks][Hkv][bs][hd]
    kp = np.zeros((40, Hkv, bs, hd), np.uint16)
    vp = np.zeros((40, Hkv, bs, hd), np.uint16)
    for lb in range(nblk):
        kp[perm[lb]] = kb[lb * bs:(lb + 1) * bs].transpose(1, 0, 2)
        vp[perm[lb]] = vb[lb * bs:(lb + 1) * bs].transpose(1, 0, 2)
    a = orc.attention_paged(q, kp, vp, Hkv * bs * hd, perm, ctx, Hq, Hkv, hd, bs, 0.125)
    b = orc.attention_contig(q, kb, vb, ctx, Hq, Hkv, hd, 0.125)
    assert np.array_equal(a, b)


def test_split_softmax_merge_equals_two_pass(orc):
    """Online softmax over splits, merged with the running-max rescaling, equals the
    oracle's two-pass result (the reordering the GPU uses)."""
    import oracle
    Hq, Hkv, hd, ctx = 4, 1, 64, 300
    k, v = _kv(90, ctx, Hkv, hd)
    kb, vb = oracle.to_bf16(k), oracle.to_bf16(v)
    kf = oracle.from_bf16(kb).reshape(ctx, hd).astype(np.float64)
    vf = oracle.from_bf16(vb).reshape(ctx, hd).astype(np.float64)
    q = synth.normal(92, Hq * hd)
    out = orc.attention_contig(q, kb, vb, ctx, Hq, Hkv, hd, 0.125).reshape(Hq, hd)
    for h in range(Hq):
        s = kf @ q[h * hd:(h + 1) * hd].astype(np.float64) * 0.125
        parts = []
        for lo in range(0, ctx, 64):
            ss = s[lo:lo + 64]
            m = ss.max()
            p = np.exp(ss - m)
            parts.append((m, p.sum(), p @ vf[lo:lo + 64]))
        M = max(m for m, _, _ in parts)
        L = sum(l * math.exp(m - M) for m, l, _ in parts)
        O = sum(o * math.exp(m - M) for m, _, o in parts) / L
        assert np.allclose(out[h], O, rtol=1e-6, atol=1e-7)


# ----------------------------------------------------------------- block pool

def test_pool_lifo_and_exhaustion(orc):
    p = orc.Pool(4, 8)
    assert [p.alloc() for _ in range(4)] == [0, 1, 2, 3]
    assert p.alloc() == -1 and p.free_count() == 0
    assert p.decref(2) == 0 and p.decref(0) == 0
    assert p.alloc() == 0 and p.alloc() == 2  # last freed, first out
    assert p.decref(7) == -1 and p.incref(-1) == -1
    for b in range(4):
        p.decref(b)
    assert p.free_count() == 4


def test_copy_on_write(orc):
    bs = 16
    p = orc.Pool(6, 32)
    a = np.array([p.alloc(), p.alloc()], np.int32)
    p.data(int(a[1]))[:] = np.arange(32, dtype=np.uint8)
    b = a.copy()  # second sequence shares both blocks
    p.incref(int(a[0]))
    p.incref(int(a[1]))
    # writing into a private block does not copy
    tmp = np.array([p.alloc()], np.int32)
    assert p.writable(tmp, 3, bs) == tmp[0]
    # writing into a shared block splits it: copy, then decref, then swap
    old = int(b[1])
    nw = p.writable(b, bs + 5, bs)
    assert nw not in (int(a[0]), int(a[1]), int(tmp[0])) and b[1] == nw
    assert np.array_equal(p.data(nw), np.arange(32, dtype=np.uint8))
    assert p.refcount(old) == 1 and p.refcount(nw) == 1
    assert b[0] == a[0] and p.refcount(int(a[0])) == 2
    p.data(nw)[0] = 99
    assert p.data(old)[0] == 0  # the other holder still reads the old contents
    # exhaustion during a split: -1, the table and the counts are left alone
    while p.alloc() >= 0:
        pass
    b2 = a.copy()
    p.incref(int(a[0]))
    assert p.writable(b2, 0, bs) == -1 and b2[0] == a[0] and p.refcount(int(a[0])) == 3


# ----------------------------------------------------------------- the model

def _tiny_model(orc, layers=None, n_blocks=16, max_pos=128, shape=synth.TINY):
    return orc.Model(shape, n_kv_blocks=n_blocks, max_pos=max_pos, layers=layers)


def test_incremental_equals_nocache(orc):
    """Decode with the paged cache equals the full no-cache recompute of the last
    position, bit for bit, with blocks in a permuted physical order."""
    m = _tiny_model(orc)
    toks = synth.TINY.tokens(20)
    bt = synth.permutation(5, 16).astype(np.int32)
    for pos, t in enumerate(toks):
        logits, best = m.decode_step(int(t), pos, bt)
    ref, rbest = m.forward_nocache(toks)
    assert np.array_equal(logits, ref) and best == rbest


def test_threads_do_not_change_a_bit(orc):
    """Spreading rows and heads over host threads keeps every output's serial sum:
    the quantisers, a GEMV and 24 decode steps give the same bits on 1 and 4 threads."""
    if orc.max_threads() < 2:
        pytest.skip("oracle built without OpenMP")
    w = synth.normal(0x7417, 300 * 688, std=0.02).reshape(300, 688)
    x = synth.normal(0x7418, 688)
    runs = []
    for n in (1, 4):
        assert orc.set_threads(n) == n
        q4 = orc.q4_0_quantize(w)
        q8, s8 = orc.i8_quantize(w)
        y = orc.gemv(orc.Mat("q4_0", q4, 300, 688), x)
        m = _tiny_model(orc)
        bt = synth.permutation(8, 16).astype(np.int32)
        for pos, t in enumerate(synth.TINY.tokens(24)):
            logits, best = m.decode_step(int(t), pos, bt)
        runs.append((q4, q8, s8, y, logits, best, m.kv().copy()))
    orc.set_threads(orc.max_threads())
    for a, b in zip(*runs):
        assert np.array_equal(np.asarray(a), np.asarray(b))


def test_paged_step_independent_of_physical_order(orc):
    toks = synth.TINY.tokens(18)
    outs = []
    for perm_seed in (None, 6, 7):
        m = _tiny_model(orc)
        bt = np.arange(16, dtype=np.int32) if perm_seed is None else synth.permutation(perm_seed, 16)
        for pos, t in enumerate(toks):
            logits, _ = m.decode_step(int(t), pos, bt)
        outs.append(logits)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_step_composition_at_position_zero(orc):
    """At position 0 attention returns v exactly, so one layer reduces to pinned parts:
    x1 = x0 + Wo bf16(v) then the MLP; checked bit for bit with distinct norm gains so
    that a swapped tensor would show."""
    import oracle
    shape = synth.TINY
    m = _tiny_model(orc, layers=1)
    d = shape.d_model
    gains = [synth.normal(100 + i, d) + 2 for i in range(3)]
    lib = oracle.lib()
    for which, g in zip((5, 6), gains[:2]):
        lib.or_model_set(m.h, which, 0, 3, g.ctypes.data, None, 1, d)
    lib.or_model_set(m.h, 102, 0, 3, gains[2].ctypes.data, None, 1, d)
    m._keep += gains
    tok = 77
    logits, best = m.decode_step(tok, 0, np.arange(16, dtype=np.int32))
    M = m.mats
    x = oracle.embed_row(M["embed"], tok)
    qkv = oracle.gemv(M["l0.qkv"], oracle.rmsnorm(x, gains[0], shape.rms_eps))
    hq = shape.n_heads * shape.head_dim
    hk = shape.n_kv_heads * shape.head_dim
    v = oracle.from_bf16(oracle.to_bf16(qkv[hq + hk:]))
    att = np.repeat(v.reshape(shape.n_kv_heads, shape.head_dim), shape.n_heads // shape.n_kv_heads, axis=0).ravel()
    x = x + oracle.gemv(M["l0.o"], att)
    xn = oracle.rmsnorm(x, gains[1], shape.rms_eps)
    a = oracle.swiglu(oracle.gemv(M["l0.gate"], xn), oracle.gemv(M["l0.up"], xn))
    x = x + oracle.gemv(M["l0.down"], a)
    ref = oracle.gemv(M["head"], oracle.rmsnorm(x, gains[2], shape.rms_eps))
    assert np.array_equal(logits, ref) and best == oracle.argmax(ref)


def test_step_composition_at_a_later_position(orc):
    """At position 20 (two blocks, a permuted table) one layer is the pinned parts
    composed, bit for bit: per position the normed input, the QKV GEMV, RoPE on q and k
    (not v) with that position's angles, K and V rounded to bf16 into the cache; then
    attention of the last q over all 21 positions with scale fp32(1/sqrt(hd)), O-proj and
    residual, the MLP and the head.  Unlike position 0 (where attention returns v), this
    fixes the rotation, the scale, the GQA head mapping and the cache positions.  The
    same composition with RoPE left out of k differs, so the check has teeth."""
    import math

    import oracle
    shape = synth.TINY
    m = _tiny_model(orc, layers=1)
    d, hd, Hq, Hkv = shape.d_model, shape.head_dim, shape.n_heads, shape.n_kv_heads
    gains = [synth.normal(200 + i, d) + 2 for i in range(3)]
    lib = oracle.lib()
    for which, g in zip((5, 6), gains[:2]):
        lib.or_model_set(m.h, which, 0, 3, g.ctypes.data, None, 1, d)
    lib.or_model_set(m.h, 102, 0, 3, gains[2].ctypes.data, None, 1, d)
    m._keep += gains
    toks = shape.tokens(21, stream=5)
    bt = synth.permutation(8, 16).astype(np.int32)
    for pos, t in enumerate(toks):
        logits, best = m.decode_step(int(t), pos, bt)

    M, eps = m.mats, shape.rms_eps
    cos, sin = oracle.rope_table(128, hd, shape.rope_theta)
    hq, hk = Hq * hd, Hkv * hd

    def compose(rope_k: bool):
        K, V = [], []
        for pos, t in enumerate(toks):
            x = oracle.embed_row(M["embed"], int(t))
            qkv = oracle.gemv(M["l0.qkv"], oracle.rmsnorm(x, gains[0], eps))
            q = oracle.rope_apply(qkv[:hq], Hq, hd, cos[pos], sin[pos])
            k = qkv[hq:hq + hk]
            if rope_k:
                k = oracle.rope_apply(k, Hkv, hd, cos[pos], sin[pos])
            K.append(oracle.to_bf16(k))
            V.append(oracle.to_bf16(qkv[hq + hk:]))
        att = oracle.attention_contig(q, np.stack(K), np.stack(V), len(toks), Hq, Hkv, hd, 1.0 / math.sqrt(hd))
        x = x + oracle.gemv(M["l0.o"], att)
        xn = oracle.rmsnorm(x, gains[1], eps)
        a = oracle.swiglu(oracle.gemv(M["l0.gate"], xn), oracle.gemv(M["l0.up"], xn))
        x = x + oracle.gemv(M["l0.down"], a)
        return oracle.gemv(M["head"], oracle.rmsnorm(x, gains[2], eps))

    ref = compose(True)
    assert np.array_equal(logits, ref) and best == oracle.argmax(ref)
    assert not np.array_equal(logits, compose(False))


def test_two_layer_composition(orc):
    """Two layers with distinct norm gains per layer, 18 positions: the step's logits
    equal the parts composed layer by layer -- every position's output of layer 0 is the
    input of layer 1, and each layer keeps its own K/V -- bit for bit.  A wrong layer
    index for a weight, a gain or a cache slice would break it."""
    import math

    import oracle
    shape = synth.TINY
    m = _tiny_model(orc, layers=2)
    d, hd, Hq, Hkv = shape.d_model, shape.head_dim, shape.n_heads, shape.n_kv_heads
    lib = oracle.lib()
    gains = {}
    for layer in range(2):
        for which in (5, 6):
            g = synth.normal(300 + 10 * layer + which, d) + 2
            lib.or_model_set(m.h, which, layer, 3, g.ctypes.data, None, 1, d)
            gains[(layer, which)] = g
    gf = synth.normal(399, d) + 2
    lib.or_model_set(m.h, 102, 0, 3, gf.ctypes.data, None, 1, d)
    m._keep += list(gains.values()) + [gf]
    toks = shape.tokens(18, stream=6)
    bt = synth.permutation(9, 16).astype(np.int32)
    for pos, t in enumerate(toks):
        logits, best = m.decode_step(int(t), pos, bt)

    M, eps = m.mats, shape.rms_eps
    cos, sin = oracle.rope_table(128, hd, shape.rope_theta)
    hq, hk = Hq * hd, Hkv * hd
    X = [oracle.embed_row(M["embed"], int(t)) for t in toks]
    for layer in range(2):
        W = {n: M[f"l{layer}.{n}"] for n in ("qkv", "o", "gate", "up", "down")}
        K, V, Q = [], [], []
        for pos, x in enumerate(X):
            qkv = oracle.gemv(W["qkv"], oracle.rmsnorm(x, gains[(layer, 5)], eps))
            Q.append(oracle.rope_apply(qkv[:hq], Hq, hd, cos[pos], sin[pos]))
            K.append(oracle.to_bf16(oracle.rope_apply(qkv[hq:hq + hk], Hkv, hd, cos[pos], sin[pos])))
            V.append(oracle.to_bf16(qkv[hq + hk:]))
        out = []
        for pos, x in enumerate(X):
            att = oracle.attention_contig(Q[pos], np.stack(K[:pos + 1]), np.stack(V[:pos + 1]), pos + 1,
                                          Hq, Hkv, hd, 1.0 / math.sqrt(hd))
            x = x + oracle.gemv(W["o"], att)
            xn = oracle.rmsnorm(x, gains[(layer, 6)], eps)
            out.append(x + oracle.gemv(W["down"], oracle.swiglu(oracle.gemv(W["gate"], xn),
                                                                 oracle.gemv(W["up"], xn))))
        X = out
    ref = oracle.gemv(M["head"], oracle.rmsnorm(X[-1], gf, eps))
    assert np.array_equal(logits, ref) and best == oracle.argmax(ref)


def test_bf16_activation_points(orc):
    """With bf16 activations (the TinyLlama workload) every GEMV input vector -- the two
    normed inputs, the attention output, the SwiGLU output and the head's normed input --
    is rounded to bf16 and nothing else is (the residual stays fp32): the step equals
    that composition bit for bit at position 9, and leaving the SwiGLU output unrounded
    differs."""
    import math
    from dataclasses import replace

    import oracle
    shape = replace(synth.TINY, act_bf16=True)
    m = orc.Model(shape, n_kv_blocks=16, max_pos=128, layers=1)
    d, hd, Hq, Hkv = shape.d_model, shape.head_dim, shape.n_heads, shape.n_kv_heads
    toks = shape.tokens(10, stream=7)
    bt = np.arange(16, dtype=np.int32)
    for pos, t in enumerate(toks):
        logits, best = m.decode_step(int(t), pos, bt)

    M, eps, ones = m.mats, shape.rms_eps, np.ones(d, np.float32)
    cos, sin = oracle.rope_table(128, hd, shape.rope_theta)
    hq, hk = Hq * hd, Hkv * hd

    def bf(v):
        return oracle.from_bf16(oracle.to_bf16(v))

    def compose(round_act: bool):
        K, V = [], []
        for pos, t in enumerate(toks):
            x = oracle.embed_row(M["embed"], int(t))
            qkv = oracle.gemv(M["l0.qkv"], bf(oracle.rmsnorm(x, ones, eps)))
            q = oracle.rope_apply(qkv[:hq], Hq, hd, cos[pos], sin[pos])
            K.append(oracle.to_bf16(oracle.rope_apply(qkv[hq:hq + hk], Hkv, hd, cos[pos], sin[pos])))
            V.append(oracle.to_bf16(qkv[hq + hk:]))
        att = oracle.attention_contig(q, np.stack(K), np.stack(V), len(toks), Hq, Hkv, hd, 1.0 / math.sqrt(hd))
        x = x + oracle.gemv(M["l0.o"], bf(att))
        xn = bf(oracle.rmsnorm(x, ones, eps))
        a = oracle.swiglu(oracle.gemv(M["l0.gate"], xn), oracle.gemv(M["l0.up"], xn))
        x = x + oracle.gemv(M["l0.down"], bf(a) if round_act else a)
        return oracle.gemv(M["head"], bf(oracle.rmsnorm(x, ones, eps)))

    ref = compose(True)
    assert np.array_equal(logits, ref) and best == oracle.argmax(ref)
    assert not np.array_equal(logits, compose(False))


@pytest.mark.parametrize("fmt", ["i8", "bf16"])
def test_tied_embedding_is_the_head_matrix(orc, fmt):
    """With tied weights (the Llama-3.2-1B shape) the token's input row is the head
    matrix's row, dequantised (int8: times its row scale): a one-layer step at position 0
    equals that composition bit for bit."""
    from dataclasses import replace

    import oracle
    shape = replace(synth.TINY, tied=True, wfmt=fmt, head_fmt=fmt)
    m = orc.Model(shape, n_kv_blocks=16, max_pos=128, layers=1)
    assert "embed" not in m.mats
    d, hd, Hq, Hkv = shape.d_model, shape.head_dim, shape.n_heads, shape.n_kv_heads
    tok = 321
    logits, best = m.decode_step(tok, 0, np.arange(16, dtype=np.int32))
    M, eps, ones = m.mats, shape.rms_eps, np.ones(d, np.float32)
    x = M["head"].dequantize()[tok].astype(np.float32)
    assert np.array_equal(x, oracle.embed_row(M["head"], tok))
    qkv = oracle.gemv(M["l0.qkv"], oracle.rmsnorm(x, ones, eps))
    v = oracle.from_bf16(oracle.to_bf16(qkv[(Hq + Hkv) * hd:]))
    att = np.repeat(v.reshape(Hkv, hd), Hq // Hkv, axis=0).ravel()
    x = x + oracle.gemv(M["l0.o"], att)
    xn = oracle.rmsnorm(x, ones, eps)
    x = x + oracle.gemv(M["l0.down"], oracle.swiglu(oracle.gemv(M["l0.gate"], xn), oracle.gemv(M["l0.up"], xn)))
    ref = oracle.gemv(M["head"], oracle.rmsnorm(x, ones, eps))
    assert np.array_equal(logits, ref) and best == oracle.argmax(ref)


def test_step_rejects_bad_arguments(orc):
    m = _tiny_model(orc)
    bt = np.arange(16, dtype=np.int32)
    with pytest.raises(ValueError):
        m.decode_step(5000, 0, bt)
    with pytest.raises(ValueError):
        m.decode_step(1, 128, bt)
    bad = bt.copy()
    bad[0] = 99
    with pytest.raises(ValueError):
        m.decode_step(1, 0, bad)


def test_slots_sharing_a_prefix_equal_independent_sequences(orc):
    """Few-slot step: three slots that borrow one 40-token prefix (two whole blocks shared,
    the half-filled third copied on write by the two borrowers) and then continue with
    their own tokens give, bit for bit, the logits of each sequence decoded alone in a
    fresh cache with its own blocks ("Mini Inference Engine", "Prefix sharing and
    copy-on-write", "Continuous batching")."""
    shape, bs = synth.TINY, synth.TINY.block_size
    n_pre, n_gen, S, max_blocks = 40, 6, 3, 8
    prefix = shape.tokens(n_pre, stream=11)
    cont = [shape.tokens(n_gen, stream=12 + s) for s in range(S)]

    m = _tiny_model(orc, n_blocks=24)
    kv = m.kv()
    tables = np.full((S, max_blocks), -1, np.int32)
    tables[0, :3] = [5, 9, 2]
    for pos, t in enumerate(prefix):
        m.decode_step(int(t), pos, tables[0])
    spare = [11, 3, 17, 20, 7, 13, 0, 22, 15]
    for s in (1, 2):
        tables[s, :3] = tables[0, :3]
        # the first write of slot s lands in the shared, half-filled block: copy, then swap
        nb = spare.pop()
        kv[nb] = kv[tables[s, 2]]
        tables[s, 2] = nb
    for s in range(S):
        tables[s, 3:5] = [spare.pop(), spare.pop()] if s else [1, 4]
    got = []
    for i in range(n_gen):
        logits, best = m.decode_step_slots([int(c[i]) for c in cont], [n_pre + i] * S, tables)
        got.append((logits.copy(), best.copy()))

    for s in range(S):
        alone = _tiny_model(orc, n_blocks=24)
        bt = np.arange(24, dtype=np.int32)
        for pos, t in enumerate(prefix):
            alone.decode_step(int(t), pos, bt)
        for i in range(n_gen):
            ref, rbest = alone.decode_step(int(cont[s][i]), n_pre + i, bt)
            assert np.array_equal(got[i][0][s], ref), (s, i)
            assert got[i][1][s] == rbest


def test_slots_sharing_without_copy_on_write_diverge(orc):
    """The copy above is needed: if a borrower writes into the shared half-filled block
    in place, the owner's later logits change (the pin would catch a missing copy)."""
    shape = synth.TINY
    n_pre = 40
    prefix = shape.tokens(n_pre, stream=11)
    m = _tiny_model(orc, n_blocks=24)
    tables = np.full((2, 8), -1, np.int32)
    tables[0, :4] = [5, 9, 2, 1]
    tables[1, :4] = [5, 9, 2, 4]  # block 2 shared, no copy
    for pos, t in enumerate(prefix):
        m.decode_step(int(t), pos, tables[0])
    a = shape.tokens(2, stream=21)
    b = shape.tokens(2, stream=22)
    m.decode_step_slots([int(a[0]), int(b[0])], [n_pre, n_pre], tables)  # both write position 40
    logits, _ = m.decode_step_slots([int(a[1]), int(b[1])], [n_pre + 1, n_pre + 1], tables)

    alone = _tiny_model(orc, n_blocks=24)
    bt = np.arange(24, dtype=np.int32)
    for pos, t in enumerate(list(prefix) + [int(a[0])]):
        alone.decode_step(int(t), pos, bt)
    ref, _ = alone.decode_step(int(a[1]), n_pre + 1, bt)
    assert not np.array_equal(logits[0], ref)


# ----------------------------------------------------------------- sampling

def _softmax(v, T):
    e = np.exp((v.astype(np.float64) - v.max()) / T)
    return e / e.sum()


def test_sampler_generator_known_answers(orc):
    """splitmix64 from its published first outputs (seed 0); the per-token uniform is
    (top 24 bits + 1/2) / 2^24 of output (pos << 32 | i)."""
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]
    assert [orc.splitmix64(0, i) for i in range(4)] == want
    assert orc.sample_uniform(0, 0, 0) == ((0xE220A8397B1DCDAF >> 40) + 0.5) / 2**24
    assert orc.sample_uniform(0, 0, 3) == ((0xF88BB8A8724C81EC >> 40) + 0.5) / 2**24
    u = np.array([orc.sample_uniform(7, p, i) for p in range(40) for i in range(50)])
    assert np.all((u > 0) & (u < 1)) and abs(u.mean() - 0.5) < 0.02


def test_sampler_greedy_limits(orc):
    """T = 0, top-k = 1 and a vanishing top-p all give the argmax, whatever the seed."""
    v = synth.normal(60, 3000)
    best = int(np.argmax(v))
    for seed in (1, 2, 3):
        assert orc.sample(v, 0.0, seed=seed, pos=5) == best
        assert orc.sample(v, 1.3, top_k=1, seed=seed, pos=5) == best
        assert orc.sample(v, 0.8, top_p=1e-9, seed=seed, pos=5) == best


def test_sampler_support(orc):
    """Every draw lies in the top-k set, and in the nucleus: the highest logits whose
    softmax mass first reaches p (computed here by numpy)."""
    v = synth.normal(61, 500)
    order = np.argsort(-v, kind="stable")
    topk = set(order[:7].tolist())
    pr = _softmax(v, 0.5)[order]
    nucleus = set(order[: int(np.searchsorted(np.cumsum(pr), 0.4)) + 1].tolist())
    for pos in range(300):
        assert orc.sample(v, 1.0, top_k=7, seed=11, pos=pos) in topk
        assert orc.sample(v, 0.5, top_p=0.4, seed=11, pos=pos) in nucleus


def test_sampler_keeps_ties_at_the_top_k_threshold(orc):
    v = np.array([3.0, 1.0, 2.0, 2.0, 2.0, 0.5], np.float32)
    seen = {orc.sample(v, 50.0, top_k=2, seed=3, pos=p) for p in range(400)}
    assert seen == {0, 2, 3, 4}


@pytest.mark.parametrize("top_k,top_p", [(0, 1.0), (3, 1.0), (0, 0.6), (4, 0.8)])
def test_sampler_frequencies_follow_the_kept_softmax(orc, top_k, top_p):
    """Over 30000 positions the draws follow q_i / sum q over the kept set (chi-square
    with 5 degrees of freedom at most, below its 99.99 % quantile 25.7)."""
    v = np.array([1.2, 0.3, -0.4, 2.0, 0.9, -1.1], np.float32)
    T = 0.9
    pr = _softmax(v, T)
    order = np.argsort(-v, kind="stable")
    keep = np.ones(v.size, bool)
    if top_k:
        keep[:] = False
        keep[order[:top_k]] = True
    if top_p < 1:
        kept_sorted = [i for i in order if keep[i]]
        mass = pr[kept_sorted] / pr[kept_sorted].sum()
        cut = int(np.searchsorted(np.cumsum(mass), top_p)) + 1
        keep[:] = False
        keep[kept_sorted[:cut]] = True
    want = np.where(keep, pr, 0.0)
    want /= want.sum()
    n = 30000
    counts = np.bincount([orc.sample(v, T, top_k=top_k, top_p=top_p, seed=0x5A, pos=p) for p in range(n)],
                         minlength=v.size)
    assert np.all(counts[~keep] == 0)
    exp_ = want[keep] * n
    chi2 = float(np.sum((counts[keep] - exp_) ** 2 / exp_))
    assert chi2 < 25.7, (counts, exp_)


def test_sampler_reproduces(orc):
    v = synth.normal(62, 2000)
    a = [orc.sample(v, 0.7, 50, 0.9, seed=99, pos=p) for p in range(30)]
    assert a == [orc.sample(v, 0.7, 50, 0.9, seed=99, pos=p) for p in range(30)]
    assert len(set(a)) > 5  # different positions draw different tokens
