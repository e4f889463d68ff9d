"""The decode step on the GPU against the oracle (teacher-forced with the oracle's tokens).

Tolerances: max |dlogit| <= 2e-2 * std(logits) per step, argmax identical wherever the
oracle's top-2 margin exceeds 1e-2; K/V cache entries within one bf16 step of the value
plus 1e-3 of the tensor's RMS (the GEMV tolerance), with > 97% of them bit-identical.
"""
import time

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


def check_logits(got, ref, pos):
    tol = 2e-2 * float(np.std(ref))
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    assert err <= tol, f"pos {pos}: max |dlogit| {err:.3e} > {tol:.3e}"


def check_argmax(got_best, ref, pos):
    top = np.sort(ref)[-2:]
    if top[1] - top[0] > 1e-2:
        assert got_best == int(np.argmax(ref)), f"pos {pos}: argmax {got_best} vs {int(np.argmax(ref))}"


PERSISTENT, CHAIN = 0, 1


def run_parity(orc, shape, layers, n_prompt, n_gen, perm_seed=5, compare_kv=True, mode=PERSISTENT):
    bs = shape.block_size
    n_tok = n_prompt + n_gen
    n_blocks = (n_tok + bs - 1) // bs + 3
    max_pos = n_blocks * bs
    om = orc.Model(shape, n_kv_blocks=n_blocks, max_pos=max_pos, layers=layers)
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos, layers=layers)
    gm.set_step_mode(mode)
    bt = synth.permutation(perm_seed, n_blocks).astype(np.int32)
    btd = torch.from_numpy(bt).cuda()
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    toks = list(prompt_tokens(shape, n_prompt))
    for pos in range(n_tok):
        ref, best = om.decode_step(int(toks[pos]), pos, bt)
        gm.decode_step(int(toks[pos]), pos, btd, logits, am)
        gm.sync()
        assert gm.step_mode == mode
        check_logits(logits.cpu().numpy(), ref, pos)
        check_argmax(int(am.item()), ref, pos)
        if pos + 1 >= len(toks):
            toks.append(best)  # teacher forcing with the oracle's greedy token
    if compare_kv:
        used = bt[: (n_tok + bs - 1) // bs]
        g = gm.kv().cpu().numpy().view(np.uint16)[used]
        r = om.kv()[used]
        gf = orc.from_bf16(g).astype(np.float64)
        rf = orc.from_bf16(r).astype(np.float64)
        # one bf16 step of the value plus the GEMV tolerance at the tensor's scale: an
        # element near zero can round to different bf16 neighbours when the fp32 GEMV
        # outputs differ by ~1e-6 of the row scale (entries past n_tok are zero on both).
        # With bf16 activations every GEMV input is rounded too: a ~1e-4 relative
        # difference in the residual flips a few percent of the rounded inputs by one
        # bf16 step (2^-8 relative), which moves later K/V values by ~1e-3 of their RMS
        # with tails several times that, hence the wider term there.
        rms = float(np.sqrt(np.mean(rf[rf != 0] ** 2)))
        err = np.abs(gf - rf)
        c, min_exact = (1e-2, 0.85) if shape.act_bf16 else (1e-3, 0.97)
        bound = np.abs(rf) * 2.0 ** -7 + c * rms
        worst = np.unravel_index(np.argmax(err / bound), err.shape)
        assert np.all(err <= bound), f"K/V {worst}: gpu {gf[worst]} oracle {rf[worst]} (rms {rms:.3g})"
        exact = float(np.mean(g == r))
        assert exact > min_exact, f"only {exact:.3f} of the K/V bf16 values are identical"
    return gm, om


@pytest.mark.parametrize("mode", [PERSISTENT, CHAIN])
def test_tiny_q4_0_prompt_and_greedy(orc, mode):
    """64 prompt tokens + 16 greedy steps of the tiny Q4_0 decoder (K = 688 ragged)."""
    run_parity(orc, synth.TINY, None, 64, 16, mode=mode)


@pytest.mark.parametrize("mode", [PERSISTENT, CHAIN])
@pytest.mark.parametrize("fmt", ["bf16", "i8", "q4_0"])
def test_llama32_shape_two_layers(orc, fmt, mode):
    """Llama-3.2-1B shapes (every GEMV and the LM head at full size), 2 of 16 layers."""
    run_parity(orc, synth.llama32_1b(fmt), 2, 5, 2, mode=mode)


@pytest.mark.parametrize("mode", [PERSISTENT, CHAIN])
@pytest.mark.parametrize("fmt,head", [("q4_g128", "q4_g128"), ("q4_g64", "i8"), ("q4_0", "q4_0")])
def test_llama32_shape_int4_groups(orc, fmt, head, mode):
    """The int4 variants of the Llama-3.2-1B shape: groups of 128 everywhere (the tied
    head and embedding too), groups of 64 with the int8 head, and Q4_0 everywhere."""
    run_parity(orc, synth.llama32_1b(fmt, head), 2, 5, 2, mode=mode)


@pytest.mark.parametrize("mode", [PERSISTENT, CHAIN])
def test_tinyllama_shape_bf16_activations(orc, mode):
    """TinyLlama shapes, Q4_0, bf16 GEMV inputs, 2 of 22 layers."""
    run_parity(orc, synth.TINYLLAMA, 2, 4, 2, mode=mode)


def test_llama32_full_depth_bf16(orc):
    """All 16 layers of the bf16 Llama-3.2-1B shape, the bench's configuration."""
    run_parity(orc, synth.LLAMA32_1B, None, 2, 1, compare_kv=False)


def test_persistent_and_chain_agree_over_long_context(orc):
    """The two step implementations compute the same arithmetic in the same order per
    row, so over 300 greedy steps their logits stay within rounding of each other
    and their tokens agree wherever the margin is clear."""
    shape = synth.TINY
    n_blocks, max_pos = 24, 24 * 16
    bt = torch.from_numpy(synth.permutation(11, n_blocks).astype(np.int32)).cuda()
    res = []
    for mode in (PERSISTENT, CHAIN):
        gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
        gm.set_step_mode(mode)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        am = torch.empty(1, dtype=torch.int32, device="cuda")
        gm.decode_step(3, 0, bt, logits, am)
        gm.decode_continue(299)
        gm.sync()
        res.append(logits.cpu().numpy())
        gm.close()
    assert np.max(np.abs(res[0] - res[1])) <= 1e-3 * float(np.std(res[1]))


@pytest.mark.parametrize("step_mode", [PERSISTENT, CHAIN])
def test_device_continuation_matches_host_steps(orc, step_mode):
    """mie_decode_continue (token and position advanced on the device) gives the same
    bits as host-driven steps fed the previous argmax."""
    shape = synth.TINY
    n_blocks, max_pos = 8, 128
    bt = torch.from_numpy(synth.permutation(9, n_blocks).astype(np.int32)).cuda()
    outs = []
    for mode in ("host", "device"):
        gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
        assert gm.step_mode == PERSISTENT  # the default where the shape is covered
        gm.set_step_mode(step_mode)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        am = torch.empty(1, dtype=torch.int32, device="cuda")
        toks = prompt_tokens(shape, 10)
        for pos, t in enumerate(toks):
            gm.decode_step(int(t), pos, bt, logits, am)
        if mode == "host":
            pos = len(toks)
            for _ in range(12):
                gm.sync()
                gm.decode_step(int(am.item()), pos, bt, logits, am)
                pos += 1
        else:
            gm.decode_continue(12)
        gm.sync()
        outs.append((logits.cpu().numpy(), int(am.item())))
        gm.close()
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    assert outs[0][1] == outs[1][1]


def test_decode_step_sync_gives_the_steps_tokens(orc):
    """mie_decode_step_sync (host token in, next token out, waiting) gives the tokens and
    logit bits of mie_decode_step followed by a read of its argmax."""
    shape = synth.TINY
    n_blocks, max_pos = 8, 128
    bt = torch.from_numpy(synth.permutation(12, n_blocks).astype(np.int32)).cuda()
    toks = [int(t) for t in prompt_tokens(shape, 6)]
    outs = []
    for sync in (False, True):
        gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        am = torch.empty(1, dtype=torch.int32, device="cuda")
        seq, tok = [], toks[0]
        for pos in range(20):
            if pos < len(toks):
                tok = toks[pos]
            if sync:
                nxt = gm.decode_step_sync(tok, pos, bt, logits)
            else:
                gm.decode_step(tok, pos, bt, logits, am)
                gm.sync()
                nxt = int(am.item())
            seq.append(nxt)
            tok = nxt
        gm.sync()
        outs.append((seq, logits.cpu().numpy()))
        gm.close()
    assert outs[0][0] == outs[1][0]
    assert np.array_equal(outs[0][1].view(np.uint32), outs[1][1].view(np.uint32))
    with pytest.raises(mie.MieError):
        gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
        try:
            gm.decode_step_sync(shape.vocab, 0, bt)  # token outside the vocabulary
        finally:
            gm.close()


@pytest.mark.parametrize("step_mode", [PERSISTENT, CHAIN])
def test_back_to_back_host_steps_without_waiting(orc, step_mode):
    """30 host-driven steps enqueued with no host wait between them (more than the ring
    of 8 pinned parameter buffers) give the bits of the same steps each followed by a
    sync, and the oracle's logits."""
    shape = synth.TINY
    n_blocks, max_pos, n = 8, 128, 30
    bt_host = synth.permutation(4, n_blocks).astype(np.int32)
    bt = torch.from_numpy(bt_host).cuda()
    toks = prompt_tokens(shape, n)
    outs = []
    for wait in (False, True):
        gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
        gm.set_step_mode(step_mode)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        am = torch.empty(1, dtype=torch.int32, device="cuda")
        for pos, t in enumerate(toks):
            gm.decode_step(int(t), pos, bt, logits, am)
            if wait:
                gm.sync()
        gm.sync()
        outs.append((logits.cpu().numpy(), int(am.item())))
        gm.close()
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    assert outs[0][1] == outs[1][1]
    om = orc.Model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
    for pos, t in enumerate(toks):
        ref, best = om.decode_step(int(t), pos, bt_host)
    check_logits(outs[0][0], ref, n - 1)
    check_argmax(outs[0][1], ref, n - 1)


def test_step_rejects_bad_inputs():
    shape = synth.TINY
    gm = build_gpu_model(shape, n_kv_blocks=4, max_pos=64)
    bt = torch.tensor([3, 1, 99, 0], dtype=torch.int32, device="cuda")
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    with pytest.raises(mie.MieError) as e:
        gm.decode_step(shape.vocab, 0, bt, logits)
    assert e.value.status == 1
    with pytest.raises(mie.MieError) as e:
        gm.decode_step(1, 64, bt, logits)
    assert e.value.status == 1
    gm.decode_step(1, 3, bt, logits)
    gm.sync()
    gm.decode_step(1, 35, bt, logits)  # block 99 is outside the 4-block pool
    with pytest.raises(mie.MieError) as e:
        gm.sync()
    assert e.value.status == 7
    gm.sync()  # the flag was cleared
    empty = mie.Model(gm.cfg)
    with pytest.raises(mie.MieError) as e:
        empty.decode_step(1, 0, bt, logits)
    assert e.value.status == 6


@pytest.mark.parametrize("phase", [1, 3, 10])
def test_bounded_wait_runs_out_then_the_step_recovers(orc, phase):
    """A phase whose input never arrives (attention, gate/up, the LM head of the tiny
    two-layer model: its input words are redirected to a buffer no phase writes) makes
    the persistent step's bounded waits give up: the step ends on its own, mie_sync
    reports MIE_E_TIMEOUT, and once the phase table is restored the same position and
    the next one match the oracle again."""
    shape = synth.TINY
    n_blocks, max_pos = 8, 128
    bt_host = synth.permutation(6, n_blocks).astype(np.int32)
    bt = torch.from_numpy(bt_host).cuda()
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
    om = orc.Model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    toks = prompt_tokens(shape, 12)
    for pos in range(10):
        om.decode_step(int(toks[pos]), pos, bt_host)
        gm.decode_step(int(toks[pos]), pos, bt, logits, am)
    gm.sync()
    assert gm.step_mode == PERSISTENT
    gm.debug_stall(phase, 1 << 14)
    t0 = time.perf_counter()
    gm.decode_step(int(toks[10]), 10, bt, logits, am)
    with pytest.raises(mie.MieError) as e:
        gm.sync()
    assert e.value.status == 5, e.value  # MIE_E_TIMEOUT
    assert time.perf_counter() - t0 < 30
    gm.debug_stall(-1)
    for pos in (10, 11):
        ref, _ = om.decode_step(int(toks[pos]), pos, bt_host)
        gm.decode_step(int(toks[pos]), pos, bt, logits, am)
        gm.sync()
        check_logits(logits.cpu().numpy(), ref, pos)
        check_argmax(int(am.item()), ref, pos)
    with pytest.raises(mie.MieError) as e:  # phase 0 has no input to withhold
        gm.debug_stall(0, 1 << 14)
    assert e.value.status == 1
    gm.close()
