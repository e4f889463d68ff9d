"""Temperature / top-k / top-p sampling on the GPU against the oracle (GPU only).

The sampler's token is an argmax of perturbed logits (Gumbel-max over the kept set), and
the uniforms behind the perturbation come from one counter-based generator that both
sides implement, so the GPU must draw the oracle's token: the two differ only where two
perturbed scores, or the top-p mass at the cut-off, tie to within fp32 rounding, which
the seeded inputs here do not produce.  Greedy (temperature 0) is the argmax, bit-exact.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

mie = pytest.importorskip("memory_bound_decode_dequant_gb300")
from memory_bound_decode_dequant_gb300.workload import build_gpu_model, prompt_tokens  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)
    mie.lib()


CASES = [(0.0, 0, 1.0), (1.0, 0, 1.0), (0.7, 50, 1.0), (0.8, 0, 0.9), (0.6, 40, 0.9), (1.3, 1000, 0.5),
         (0.9, 1, 1.0), (2.0, 0, 0.05)]


@pytest.mark.parametrize("T,top_k,top_p", CASES)
def test_sample_matches_oracle(orc, T, top_k, top_p):
    """128,256 logits (the Llama-3.2-1B vocabulary), 12 positions and two seeds each."""
    V = 128256
    ws = torch.empty(mie.mie_sample_workspace_bytes(), dtype=torch.uint8, device="cuda")
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    for case in range(3):
        v = synth.normal(7000 + case, V) * np.float32(2.0)
        vd = torch.from_numpy(v).cuda()
        for seed in (0x5EED, 2**63 + 17):
            for pos in (0, 1, 2, 127, 128, 129, 511, 2047, 4000, 10**6, 2**31 - 1, 77):
                mie.mie_sample(vd, T, top_k, top_p, seed, pos, out, ws)
                got = int(out.item())
                want = orc.sample(v, T, top_k, top_p, seed, pos)
                assert got == want, (case, seed, pos, got, want)
    if T == 0.0:
        assert got == int(np.argmax(v))


def test_sample_is_reproducible_and_uses_the_seed(orc):
    v = torch.from_numpy(synth.normal(7100, 32000)).cuda()
    a = [int(mie.mie_sample(v, 0.8, 0, 0.95, 11, p).item()) for p in range(16)]
    b = [int(mie.mie_sample(v, 0.8, 0, 0.95, 11, p).item()) for p in range(16)]
    c = [int(mie.mie_sample(v, 0.8, 0, 0.95, 12, p).item()) for p in range(16)]
    assert a == b and a != c


def test_sample_small_vocab_and_edges(orc):
    """n = 1 and n smaller than one CTA's share; top_k >= n keeps all; ties at the top-k
    threshold are all kept."""
    for v in (np.array([0.25], np.float32), synth.normal(7200, 37), np.array([3, 1, 2, 2, 2, 0.5], np.float32)):
        vd = torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda()
        for (T, k, p) in [(1.0, 0, 1.0), (50.0, 2, 1.0), (0.5, 100, 0.7), (1.0, 3, 0.3)]:
            for pos in range(20):
                got = int(mie.mie_sample(vd, T, k, p, 3, pos).item())
                assert got == orc.sample(v, T, k, p, 3, pos)
    with pytest.raises(mie.MieError):
        mie.mie_sample(vd, 1.0, -1, 1.0, 0, 0)
    with pytest.raises(mie.MieError):
        mie.mie_sample(vd, 1.0, 0, 0.0, 0, 0)


def test_sampled_steps_follow_the_oracle(orc):
    """The tiny decoder with sampling inside its graph (persistent step + sampler),
    teacher-forced with the oracle's draws: each step's token is the oracle's draw from
    the oracle's logits at the same (seed, position)."""
    shape = synth.TINY
    n_blocks, max_pos = 8, 128
    T, top_k, top_p, seed = 0.7, 40, 0.9, 0xC0FFEE
    bt_host = synth.permutation(12, n_blocks).astype(np.int32)
    bt = torch.from_numpy(bt_host).cuda()
    om = orc.Model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
    gm.set_sampling(T, top_k, top_p, seed)
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    tok = int(prompt_tokens(shape, 1)[0])
    drawn = 0
    for pos in range(24):
        ref_logits, _ = om.decode_step(tok, pos, bt_host)
        want = orc.sample(ref_logits, T, top_k, top_p, seed, pos)
        gm.decode_step(tok, pos, bt, logits, am)
        gm.sync()
        assert int(am.item()) == want, pos
        drawn += want != int(np.argmax(ref_logits))
        tok = want
    assert drawn > 0  # the draws are not just the argmax
    gm.close()


def test_sampled_continuation_matches_host_steps(orc):
    """mie_decode_continue with sampling (the sampler advances token and position on the
    device) draws the same tokens as host-driven sampled steps, and another seed draws
    others."""
    shape = synth.TINY
    n_blocks, max_pos = 8, 128
    bt = torch.from_numpy(synth.permutation(13, n_blocks).astype(np.int32)).cuda()
    runs = []
    for mode, seed in (("host", 5), ("device", 5), ("device", 6)):
        gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
        gm.set_sampling(1.0, 0, 0.95, seed)
        am = torch.empty(1, dtype=torch.int32, device="cuda")
        toks = []
        gm.decode_step(17, 0, bt, None, am)
        if mode == "host":
            for pos in range(1, 20):
                gm.sync()
                toks.append(int(am.item()))
                gm.decode_step(toks[-1], pos, bt, None, am)
            gm.sync()
            toks.append(int(am.item()))
        else:
            gm.sync()
            toks.append(int(am.item()))
            for _ in range(19):
                gm.decode_continue(1)
                gm.sync()
                toks.append(int(am.item()))
        runs.append(toks)
        gm.close()
    assert runs[0] == runs[1]
    assert runs[0] != runs[2]
