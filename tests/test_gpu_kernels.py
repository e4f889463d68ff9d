"""Parity of the CUDA kernels with the oracle, through the C ABI (GPU only).

Tolerances (the arithmetic fixes them):
  * quantisers, K/V gathers, argmax: bit-exact;
  * GEMV: |dy_i| <= 1e-3 * max(|y_ref_i|, rms(y_ref)) (fp32 accumulation in another
    order than the oracle's fp64 sum);
  * attention: |do| <= 1e-4 * max(|o_ref|, rms(o_ref)) + 1e-6 (fp32 online softmax
    against the fp64 two-pass softmax over the same bf16 K/V).
"""
import math

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

mie = pytest.importorskip("memory_bound_decode_dequant_gb300")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)
    mie.lib()
    yield
    mie.mie_check()


def gemv_close(y, ref):
    ref = ref.astype(np.float64)
    rms = math.sqrt(float(np.mean(ref ** 2))) if ref.size else 0.0
    tol = 1e-3 * np.maximum(np.abs(ref), rms)
    err = np.abs(y.astype(np.float64) - ref)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, f"{bad.size} rows out of tolerance, worst {float((err / np.maximum(tol, 1e-30)).max()):.3g}x"


def bf16_vector(orc, seed, n):
    return orc.from_bf16(orc.to_bf16(synth.normal(seed, n)))


# ------------------------------------------------------------------ quantisers

@pytest.mark.parametrize("shape", [(1, 1), (3, 40), (64, 688), (257, 2048), (16384, 2048)])
def test_quantizers_bit_exact(orc, shape):
    M, K = shape
    w = synth.normal(1000 + M + K, M * K, std=0.02).reshape(M, K)
    w[0, : min(K, 32)] = 0.0  # a zero block / partly zero row
    wd = torch.from_numpy(w).cuda()
    q4 = mie.mie_quantize_q4_0(wd)
    qi, si = mie.mie_quantize_i8(wd)
    b16 = mie.mie_convert_bf16(wd)
    torch.cuda.synchronize()
    assert np.array_equal(q4.cpu().numpy(), orc.q4_0_quantize(w))
    rq, rs = orc.i8_quantize(w)
    assert np.array_equal(qi.cpu().numpy(), rq)
    assert np.array_equal(si.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(b16.view(torch.int16).cpu().numpy().view(np.uint16), orc.to_bf16(w))


@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("shape", [(1, 1), (3, 40), (64, 688), (257, 2048), (4096, 8192)])
def test_q4_group_quantizer_bit_exact(orc, group, shape):
    """4-bit groups of 64 / 128 (ragged rows zero-padded) quantise to the oracle's bytes."""
    M, K = shape
    w = synth.normal(1100 + M + K + group, M * K, std=0.02).reshape(M, K)
    w[0, : min(K, group)] = 0.0  # a zero group
    got = mie.mie_quantize_q4(torch.from_numpy(w).cuda(), group)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), orc.q4_quantize(w, group))


@pytest.mark.parametrize("group", [64, 128])
def test_q4_group_pack_layout(orc, group):
    """The GPU layout holds the groups' 16-byte sub-blocks in row order and one scale per
    group, the scale rows padded to a multiple of 8."""
    M, K = 5, 300
    w = synth.normal(78, M * K, std=0.02).reshape(M, K)
    groups = orc.q4_quantize(w, group)
    ng = groups.shape[1]
    nb, ngp = ng * group // 32, (ng + 7) // 8 * 8
    packed = mie.mie_q4_pack(torch.from_numpy(groups).cuda(), M, K, group).cpu().numpy()
    assert packed.size == mie.mie_q4_packed_bytes(M, K, group)
    nib = packed[: M * nb * 16].reshape(M, nb, 16)
    off = ((M * nb * 16 + 255) // 256) * 256
    sc = packed[off: off + M * ngp * 2].view(np.uint16).reshape(M, ngp)
    assert np.array_equal(nib, groups[:, :, 2:].reshape(M, ng, group // 32, 16).reshape(M, nb, 16))
    assert np.array_equal(sc[:, :ng], groups[:, :, 0].astype(np.uint16) | (groups[:, :, 1].astype(np.uint16) << 8))
    assert np.all(sc[:, ng:] == 0)


def test_q4_0_pack_layout(orc):
    """The GPU layout holds the canonical nibbles and scales, plane by plane."""
    M, K = 5, 70
    w = synth.normal(77, M * K, std=0.02).reshape(M, K)
    blocks = orc.q4_0_quantize(w)
    packed = mie.mie_q4_0_pack(torch.from_numpy(blocks).cuda(), M, K).cpu().numpy()
    nb, nbp = 3, 8  # scale rows padded to a multiple of 8
    nib = packed[: M * nb * 16].reshape(M, nb, 16)
    off = ((M * nb * 16 + 255) // 256) * 256
    sc = packed[off: off + M * nbp * 2].view(np.uint16).reshape(M, nbp)
    assert np.array_equal(nib, blocks[:, :, 2:])
    assert np.array_equal(sc[:, :nb], blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
    assert np.all(sc[:, nb:] == 0)


# ------------------------------------------------------------------ GEMV

def _gemv_both(orc, fmt, M, K, seed, rows=None, x=None):
    """GPU GEMV over the full matrix; oracle over `rows` (all when None)."""
    w = synth.normal(seed, M * K, std=0.02).reshape(M, K)
    if x is None:
        x = bf16_vector(orc, seed + 1, K)
    wd = torch.from_numpy(w).cuda()
    xd = torch.from_numpy(x).cuda()
    if fmt == "bf16":
        y = mie.mie_gemv_bf16(mie.mie_convert_bf16(wd), xd)
    elif fmt == "i8":
        q, s = mie.mie_quantize_i8(wd)
        y = mie.mie_gemv_i8(q, s, xd)
    elif fmt == "q4_0":
        y = mie.mie_gemv_q4_0(mie.mie_q4_0_pack(mie.mie_quantize_q4_0(wd), M, K), xd, M, K)
    else:
        g = mie.Q4_GROUP[fmt]
        y = mie.mie_gemv_q4(mie.mie_q4_pack(mie.mie_quantize_q4(wd, g), M, K, g), g, xd, M, K)
    del wd
    y = y.cpu().numpy()
    sel = np.arange(M) if rows is None else rows
    ref = orc.gemv(orc.Mat.quantize(fmt, w[sel]), x)
    return y[sel], ref


@pytest.mark.parametrize("fmt", ["bf16", "i8", "q4_0", "q4_g64", "q4_g128"])
@pytest.mark.parametrize("shape", [(1, 32), (7, 48), (33, 688), (300, 2048), (1000, 8192), (77, 5632),
                                   (5, 16384), (2049, 256)])
def test_gemv_small_and_ragged(orc, fmt, shape):
    M, K = shape
    y, ref = _gemv_both(orc, fmt, M, K, 2000 + M + K)
    gemv_close(y, ref)


@pytest.mark.parametrize("fmt", ["q4_0", "q4_g64", "q4_g128"])
@pytest.mark.parametrize("K", [1, 31, 33, 40, 100, 129, 200])
def test_gemv_q4_0_any_k(orc, fmt, K):
    y, ref = _gemv_both(orc, fmt, 9, K, 3000 + K)
    gemv_close(y, ref)


@pytest.mark.parametrize("fmt", ["bf16", "i8", "q4_0", "q4_g64", "q4_g128"])
@pytest.mark.parametrize("xscale", [1e-30, 1e-12, 1e12, 1e30, "mixed"])
@pytest.mark.parametrize("K", [688, 4096])
def test_gemv_input_magnitudes(orc, fmt, xscale, K):
    """Inputs far from unit size: the int8 / Q4_0 dot products scale their input registers
    by a power of two chosen from each group's largest |x|, so tiny and huge vectors
    (and a group holding 1e4 beside 1e-4) keep full precision."""
    x = bf16_vector(orc, 7000 + K, K)
    if xscale == "mixed":
        x = (x * 1e-4).astype(np.float32)
        x[::32] = 1e4
    else:
        x = (x * np.float32(xscale)).astype(np.float32)
    y, ref = _gemv_both(orc, fmt, 65, K, 7100 + K, x=x)
    assert np.all(np.isfinite(y))
    gemv_close(y, ref)


@pytest.mark.parametrize("fmt", ["bf16", "i8", "q4_0", "q4_g128"])
@pytest.mark.parametrize("name,M,K", synth.SWEEP_GEMV)
def test_gemv_full_size_sampled_rows(orc, fmt, name, M, K):
    """Llama-3.2-1B decode shapes; the oracle checks 256 sampled rows plus the first and
    last, the GPU computes every row in the launch configuration the sweep times."""
    rows = np.unique(np.concatenate([[0, M - 1], synth.uniform_int(4000 + M, 256, 0, M)]))
    y, ref = _gemv_both(orc, fmt, M, K, 5000 + M + K, rows)
    gemv_close(y, ref)


def test_gemv_rejects_aliasing_and_bad_k():
    x = torch.zeros(64, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mie.MieError):
        mie.mie_gemv_bf16(W, x, x)
    with pytest.raises(mie.MieError):
        mie.mie_gemv_bf16(torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda"), torch.zeros(12, device="cuda"))


# ------------------------------------------------------------------ attention

def _pool(orc, seed, n_blocks, Hkv, bs, hd):
    k = synth.normal(seed, n_blocks * Hkv * bs * hd).reshape(n_blocks, Hkv, bs, hd)
    v = synth.normal(seed + 1, n_blocks * Hkv * bs * hd).reshape(n_blocks, Hkv, bs, hd)
    return orc.to_bf16(k), orc.to_bf16(v)


def _attn_gpu(q, kp, vp, stride, n_pool, bt, ctx, Hq, Hkv, hd, bs, scale):
    kd = torch.from_numpy(kp.view(np.int16)).cuda()
    vd = torch.from_numpy(vp.view(np.int16)).cuda()
    out = mie.mie_paged_attn_decode(torch.from_numpy(q).cuda(), kd, vd, stride, n_pool,
                                    torch.from_numpy(bt).cuda(), ctx, Hq, Hkv, hd, bs, scale)
    return out.cpu().numpy()


def attn_close(out, ref):
    ref = ref.astype(np.float64)
    rms = math.sqrt(float(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(out - ref)
    assert np.all(err <= 1e-4 * np.maximum(np.abs(ref), rms) + 1e-6), float(err.max())


@pytest.mark.parametrize("Hq,Hkv,hd", [(32, 8, 64), (8, 2, 32), (32, 4, 64), (16, 16, 128), (8, 1, 128)])
@pytest.mark.parametrize("ctx", [1, 5, 16, 17, 100, 512, 2048])
def test_paged_attention(orc, Hq, Hkv, hd, ctx):
    bs = 16
    nblk = (ctx + bs - 1) // bs
    n_pool = nblk + 7
    kp, vp = _pool(orc, 6000 + ctx + hd, n_pool, Hkv, bs, hd)
    bt = synth.permutation(6100 + ctx, n_pool)[:nblk].astype(np.int32)
    q = synth.normal(6200 + ctx, Hq * hd)
    scale = float(np.float32(1 / math.sqrt(hd)))
    stride = Hkv * bs * hd
    out = _attn_gpu(q, kp, vp, stride, n_pool, bt, ctx, Hq, Hkv, hd, bs, scale)
    ref = orc.attention_paged(q, kp, vp, stride, bt, ctx, Hq, Hkv, hd, bs, scale)
    attn_close(out, ref)


@pytest.mark.parametrize("ctx", [512, 2048, 8192])
def test_paged_attention_sweep_shapes(orc, ctx):
    """The sweep's 32q/8kv heads, head_dim 64, randomly permuted physical blocks, with a
    pool laid out like the model's ([blocks][layers][k|v][Hkv][16][hd], layer 1 of 2)."""
    Hq, Hkv, hd, bs, L = 32, 8, 64, 16, 2
    nblk = ctx // bs
    n_pool = nblk + 3
    raw = synth.normal(7000 + ctx, n_pool * L * 2 * Hkv * bs * hd).reshape(n_pool, L, 2, Hkv, bs, hd)
    pool = orc.to_bf16(raw)
    bt = synth.permutation(7100 + ctx, n_pool)[:nblk].astype(np.int32)
    q = synth.normal(7200 + ctx, Hq * hd)
    stride = L * 2 * Hkv * bs * hd
    flat = pool.reshape(-1)
    kbase = flat[Hkv * bs * hd * 2:]            # layer 1, k
    vbase = flat[Hkv * bs * hd * 3:]            # layer 1, v
    pd = torch.from_numpy(flat.view(np.int16)).cuda()
    kd = pd[Hkv * bs * hd * 2:]
    vd = pd[Hkv * bs * hd * 3:]
    out = mie.mie_paged_attn_decode(torch.from_numpy(q).cuda(), kd, vd, stride, n_pool, torch.from_numpy(bt).cuda(),
                                    ctx, Hq, Hkv, hd, bs, 0.125).cpu().numpy()
    ref = orc.attention_paged(q, kbase, vbase, stride, bt, ctx, Hq, Hkv, hd, bs, 0.125)
    attn_close(out, ref)


def test_attention_gather_is_bit_exact(orc):
    """The same K/V bytes in two different physical orders give identical output bits."""
    Hq, Hkv, hd, bs, ctx = 32, 8, 64, 16, 300
    nblk = (ctx + bs - 1) // bs
    kp, vp = _pool(orc, 8000, nblk, Hkv, bs, hd)
    perm = synth.permutation(8001, nblk + 5)[:nblk].astype(np.int32)
    kp2 = np.zeros((nblk + 5,) + kp.shape[1:], np.uint16)
    vp2 = np.zeros_like(kp2)
    kp2[perm] = kp
    vp2[perm] = vp
    q = synth.normal(8002, Hq * hd)
    stride = Hkv * bs * hd
    a = _attn_gpu(q, kp, vp, stride, nblk, np.arange(nblk, dtype=np.int32), ctx, Hq, Hkv, hd, bs, 0.125)
    b = _attn_gpu(q, kp2, vp2, stride, nblk + 5, perm, ctx, Hq, Hkv, hd, bs, 0.125)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_attention_edge_cases(orc):
    Hq, Hkv, hd, bs = 8, 2, 32, 16
    kp, vp = _pool(orc, 9000, 4, Hkv, bs, hd)
    q = synth.normal(9001, Hq * hd)
    bt = np.array([2, 0, 3, 1], np.int32)
    # empty context -> zeros
    out = _attn_gpu(q, kp, vp, Hkv * bs * hd, 4, bt, 0, Hq, Hkv, hd, bs, 0.17)
    assert np.all(out == 0)
    # ctx 1 -> v_0 exactly
    out = _attn_gpu(q, kp, vp, Hkv * bs * hd, 4, bt, 1, Hq, Hkv, hd, bs, 0.17).reshape(Hq, hd)
    v0 = orc.from_bf16(vp[2, :, 0, :])
    for h in range(Hq):
        assert np.array_equal(out[h], v0[h // 4])


@pytest.mark.parametrize("Hq,Hkv,hd", [(32, 8, 64), (16, 8, 64), (64, 8, 64), (8, 1, 128)])
@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("ctx", [1, 23, 300, 777])
def test_paged_attention_tensor_core_block_sizes(orc, Hq, Hkv, hd, bs, ctx):
    """The tensor-core kernel (head_dim 64 / 128) with 8- and 32-token blocks: one 2-D
    tensor copy per block, splits whose token count is no multiple of 16, and group
    sizes 2, 4 and 8 (two 16-row tiles)."""
    nblk = (ctx + bs - 1) // bs
    n_pool = nblk + 3
    kp, vp = _pool(orc, 6500 + ctx + bs, n_pool, Hkv, bs, hd)
    bt = synth.permutation(6600 + ctx + bs, n_pool)[:nblk].astype(np.int32)
    q = synth.normal(6700 + ctx + hd, Hq * hd)
    scale = float(np.float32(1 / math.sqrt(hd)))
    stride = Hkv * bs * hd
    out = _attn_gpu(q, kp, vp, stride, n_pool, bt, ctx, Hq, Hkv, hd, bs, scale)
    ref = orc.attention_paged(q, kp, vp, stride, bt, ctx, Hq, Hkv, hd, bs, scale)
    attn_close(out, ref)


@pytest.mark.parametrize("hd", [64, 128])
def test_attention_edge_cases_tensor_core(orc, hd):
    """Empty context gives zeros; a one-token context gives v_0 exactly (P = 1 in the
    first bf16 plane, zero in the others)."""
    Hq, Hkv, bs = 8, 2, 16
    kp, vp = _pool(orc, 9200 + hd, 4, Hkv, bs, hd)
    q = synth.normal(9201, Hq * hd)
    bt = np.array([2, 0, 3, 1], np.int32)
    out = _attn_gpu(q, kp, vp, Hkv * bs * hd, 4, bt, 0, Hq, Hkv, hd, bs, 0.17)
    assert np.all(out == 0)
    out = _attn_gpu(q, kp, vp, Hkv * bs * hd, 4, bt, 1, Hq, Hkv, hd, bs, 0.17).reshape(Hq, hd)
    v0 = orc.from_bf16(vp[2, :, 0, :])
    for h in range(Hq):
        assert np.array_equal(out[h], v0[h // 4])


def test_attention_stride_not_a_row_multiple(orc):
    """A block stride that is no multiple of head_dim cannot be read as rows of a 2-D
    tensor; the kernel of bulk copies serves it, with the same results."""
    Hq, Hkv, hd, bs, ctx = 32, 8, 64, 16, 200
    nblk = (ctx + bs - 1) // bs
    stride = Hkv * bs * hd + 8
    raw_k = synth.normal(9300, nblk * stride + 8)
    raw_v = synth.normal(9301, nblk * stride + 8)
    kp, vp = orc.to_bf16(raw_k), orc.to_bf16(raw_v)
    bt = synth.permutation(9302, nblk).astype(np.int32)
    q = synth.normal(9303, Hq * hd)
    out = _attn_gpu(q, kp, vp, stride, nblk, bt, ctx, Hq, Hkv, hd, bs, 0.125)
    ref = orc.attention_paged(q, kp, vp, stride, bt, ctx, Hq, Hkv, hd, bs, 0.125)
    attn_close(out, ref)


@pytest.mark.parametrize("hd", [32, 64])
def test_attention_bad_block_id_latches_error_any_kernel(orc, hd):
    Hq, Hkv, bs = 8, 2, 16
    kp, vp = _pool(orc, 9400 + hd, 4, Hkv, bs, hd)
    q = synth.normal(9401, Hq * hd)
    mie.mie_check()
    bt = np.array([1, 9, 0], np.int32)  # 9 is outside the 4-block pool
    _attn_gpu(q, kp, vp, Hkv * bs * hd, 4, bt, 40, Hq, Hkv, hd, bs, 0.17)
    with pytest.raises(mie.MieError) as e:
        mie.mie_check()
    assert e.value.status == 7
    mie.mie_check()


def test_attention_bad_block_id_latches_error(orc):
    Hq, Hkv, hd, bs = 8, 2, 32, 16
    kp, vp = _pool(orc, 9100, 4, Hkv, bs, hd)
    q = synth.normal(9101, Hq * hd)
    mie.mie_check()
    bt = np.array([1, 9, 0], np.int32)  # 9 is outside the 4-block pool
    _attn_gpu(q, kp, vp, Hkv * bs * hd, 4, bt, 40, Hq, Hkv, hd, bs, 0.17)
    with pytest.raises(mie.MieError) as e:
        mie.mie_check()
    assert e.value.status == 7
    mie.mie_check()  # cleared


# ------------------------------------------------------------------ argmax

@pytest.mark.parametrize("n", [1, 7, 1000, 4097, 32000, 128256])
def test_argmax(orc, n):
    v = synth.normal(10000 + n, n)
    got = int(mie.mie_argmax(torch.from_numpy(v).cuda()).item())
    assert got == orc.argmax(v)


def test_argmax_ties_pick_lowest_index(orc):
    v = synth.normal(10500, 128256)
    m = v.max() + 1
    v[[90000, 7, 128255, 5000]] = m
    assert int(mie.mie_argmax(torch.from_numpy(v).cuda()).item()) == 7 == orc.argmax(v)
    v = np.zeros(50000, np.float32)
    assert int(mie.mie_argmax(torch.from_numpy(v).cuda()).item()) == 0


@pytest.mark.parametrize("load_bytes", [16, 32])
@pytest.mark.parametrize("blocks_per_sm", [1, 2, 4])
def test_hbm_read_probe_reads_every_word_once(load_bytes, blocks_per_sm):
    """The probe's XOR of all 32-bit words equals numpy's, on buffers that end in a
    ragged part of the grid stride and on one single load."""
    for n_words in ((1 << 22) + 8 * 37, load_bytes // 4):
        words = synth.uniform_int(0x5052 + n_words, n_words, -(1 << 31), (1 << 31) - 1)
        want = int(np.bitwise_xor.reduce(words.view(np.uint32)))
        d = torch.from_numpy(words).cuda()
        got = mie.mie_hbm_read_probe(d, load_bytes=load_bytes, blocks_per_sm=blocks_per_sm)
        torch.cuda.synchronize()
        assert (int(got.item()) & 0xFFFFFFFF) == want, (n_words, load_bytes, blocks_per_sm)
