"""The allocation-free attention entry point, through the C ABI (GPU only).

mie_paged_attn_decode_noalloc is for callers that cannot allocate device memory when
they run attention, so they cannot pass a workspace: it keeps its partial results in an
array built into the library.  Here two calls in a row (the second reusing the array
the first left behind, with a different context length and split count) must give the
same bits as the workspace entry point on the same inputs -- both run the same kernel
with the same split count and merge order, so any difference would mean a corrupted
read of the shared array -- and both must match the oracle within the attention
tolerance of the other kernel tests.  This file sorts last so a stopping run has
already run every other test; it also passes on its own in a fresh process.
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


def _case(seed, ctx, Hq=32, Hkv=8, hd=64, bs=16):
    nblk = (ctx + bs - 1) // bs
    n_pool = nblk + 5
    k = synth.normal(seed, n_pool * Hkv * bs * hd)
    v = synth.normal(seed + 1, n_pool * Hkv * bs * hd)
    kd = torch.from_numpy(k).cuda().to(torch.bfloat16).view(torch.int16)
    vd = torch.from_numpy(v).cuda().to(torch.bfloat16).view(torch.int16)
    q = torch.from_numpy(synth.normal(seed + 2, Hq * hd)).cuda()
    bt = torch.from_numpy(synth.permutation(seed + 3, n_pool)[:nblk].astype(np.int32)).cuda()
    return dict(q=q, k_pool=kd, v_pool=vd, block_stride=Hkv * bs * hd, n_pool_blocks=n_pool, block_table=bt,
                ctx_len=ctx, Hq=Hq, Hkv=Hkv, hd=hd, bs=bs, scale=1.0 / math.sqrt(hd))


def _close(out, ref):
    out = out.cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = math.sqrt(float(np.mean(ref ** 2)))
    assert np.all(np.abs(out - ref) <= 1e-4 * np.maximum(np.abs(ref), rms) + 1e-6)


def _oracle(orc, c):
    return orc.attention_paged(c["q"].cpu().numpy(), c["k_pool"].cpu().numpy().view(np.uint16),
                               c["v_pool"].cpu().numpy().view(np.uint16), c["block_stride"],
                               c["block_table"].cpu().numpy(), c["ctx_len"], c["Hq"], c["Hkv"], c["hd"],
                               c["bs"], c["scale"])


def test_no_alloc_matches_workspace_entry_on_two_calls_in_a_row(orc):
    for seed, ctx in ((900, 2048), (910, 300)):
        c = _case(seed, ctx)
        ref = mie.mie_paged_attn_decode(**c)
        got = mie.mie_paged_attn_decode_noalloc(**c)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), f"ctx {ctx}: not bit-identical"
        want = _oracle(orc, c)
        _close(ref, want)
        _close(got, want)
    mie.mie_check()


def test_no_alloc_rejects_sizes_beyond_its_array():
    # one KV head of group 8 and head_dim 128 over 5000 tokens needs ~1.3 MB of scratch
    need = mie.mie_paged_attn_workspace_bytes(8, 1, 128, 5000, 16)
    assert need > (1 << 20)
    c = _case(920, 64, Hq=8, Hkv=1, hd=128)
    c["ctx_len"] = 5000
    c["block_table"] = torch.zeros(5000 // 16 + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(mie.MieError) as e:
        mie.mie_paged_attn_decode_noalloc(**c)
    assert e.value.status == 2 and "scratch" in str(e.value)
