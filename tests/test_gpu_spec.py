"""Verify passes and speculative greedy decoding on the GPU (GPU only).

The Rust page's speculative decoding rests on one property: a batched pass over several
positions gives exactly the bits of single-position passes, so greedy output with
speculation equals greedy output without it, token for token.  Here the batched pass is
mie_verify_step (k positions of one sequence as k slots of the few-slot kernels), and:
  * its logits equal those of k one-position passes, bit for bit;
  * mie_generate gives the same tokens with and without prompt-lookup speculation on a
    prompt that repeats itself (so the lookup proposes guesses);
  * its tokens are the oracle's greedy tokens (teacher-forced comparison of the logits
    at the argmax tolerance: identical wherever the oracle's top-2 margin exceeds 1e-2).
"""
from dataclasses import replace

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


def _run_passes(gm, shape, toks, bt, k):
    """Positions 0 .. len(toks)-1 in passes of k positions; the logits of every position."""
    n = len(toks)
    out = np.zeros((n, shape.vocab), np.float32)
    logits = torch.empty((k, shape.vocab), dtype=torch.float32, device="cuda")
    for p0 in range(0, n, k):
        m = min(k, n - p0)
        gm.verify_step(toks[p0:p0 + m], p0, bt, logits[:m])
        gm.sync()
        out[p0:p0 + m] = logits[:m].cpu().numpy()
    return out


@pytest.mark.parametrize("fmt", ["bf16", "i8", "q4_g128"])
def test_verify_pass_equals_single_position_passes(orc, fmt):
    shape = replace(synth.TINY, wfmt=fmt, head_fmt=fmt)
    n_blocks, n = 8, 37
    bt = torch.from_numpy(synth.permutation(21, n_blocks).astype(np.int32)).cuda()
    toks = [int(t) for t in prompt_tokens(shape, n)]
    ref = None
    for k in (1, 3, 4, 8):
        gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * 16, max_slots=8)
        got = _run_passes(gm, shape, toks, bt, k)
        gm.close()
        if ref is None:
            ref = got
        else:
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"k = {k}"


def test_verify_pass_equals_single_position_passes_llama32_width(orc):
    """The Llama-3.2-1B widths (K = 2048 / 8192 slices, the 128256-row head), 1 layer."""
    shape = replace(synth.llama32_1b("bf16"), n_layers=1)
    n_blocks, n = 4, 12
    bt = torch.from_numpy(synth.permutation(22, n_blocks).astype(np.int32)).cuda()
    toks = [int(t) for t in prompt_tokens(shape, n)]
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * 16, max_slots=4)
    a = _run_passes(gm, shape, toks, bt, 1)
    b = _run_passes(gm, shape, toks, bt, 4)
    gm.close()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def _repetitive_prompt(shape, period=12, repeats=4):
    base = [int(t) for t in prompt_tokens(shape, period, stream=5)]
    return base * repeats


def test_speculative_generation_equals_plain_generation(orc):
    shape = replace(synth.TINY, wfmt="bf16", head_fmt="bf16")
    n_blocks = 12
    bt = torch.from_numpy(synth.permutation(23, n_blocks).astype(np.int32)).cuda()
    prompt = _repetitive_prompt(shape)
    outs, stats = [], []
    for spec in (1, 4):
        gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * 16, max_slots=8)
        toks, st = gm.generate(prompt, 60, bt, spec_max=spec)
        gm.close()
        outs.append(toks)
        stats.append(st)
    assert np.array_equal(outs[0], outs[1])
    assert stats[0]["proposed"] == 0 and stats[1]["proposed"] > 0
    assert stats[1]["passes"] <= stats[0]["passes"]


def test_generation_matches_the_oracle_greedy_tokens(orc):
    """mie_generate's tokens against the oracle's greedy decode of the same prompt: equal
    up to the first position where the oracle's top-2 margin is 1e-2 or less."""
    shape = synth.TINY
    n_blocks = 10
    bt_host = synth.permutation(25, n_blocks).astype(np.int32)
    bt = torch.from_numpy(bt_host).cuda()
    prompt = [int(t) for t in prompt_tokens(shape, 20, stream=7)]
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * 16, max_slots=8)
    toks, _ = gm.generate(prompt, 30, bt, spec_max=4)
    gm.close()
    om = orc.Model(shape, n_kv_blocks=n_blocks, max_pos=n_blocks * 16)
    seq = list(prompt)
    for pos in range(len(prompt) + 30 - 1):
        logits, best = om.decode_step(seq[pos], pos, bt_host)
        if pos >= len(prompt) - 1:
            top = np.sort(logits)[-2:]
            if top[1] - top[0] <= 1e-2:
                break  # a near tie: later tokens may differ legitimately
            assert int(toks[pos - len(prompt) + 1]) == best, pos
            if pos + 1 >= len(seq):
                seq.append(best)
