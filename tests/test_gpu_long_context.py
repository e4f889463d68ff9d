"""The decode step at the bench's shapes and long contexts, against the oracle.

The K/V cache of both sides is filled with the same seeded N(0, 1) bf16 values (a
synthetic prefill: the step's arithmetic does not depend on where cached values came
from), so positions far into the context are reached without running thousands of
oracle steps.  Each case then runs two teacher-forced steps at several positions,
through a permuted block table, in the same kernel instantiation the bench times:

  * Llama-3.2-1B shape (full-width GEMVs and the 128256-row LM head, 2 of 16 layers),
    bf16 / int8 / Q4_0 layers with the int8 head: positions 150, 600 and 2100, where
    the persistent step's attention runs 1, 3 and 9 splits of 256 tokens and merges
    them; bf16 also at 8250, past the 512 block ids the step stages in shared memory.
  * TinyLlama shape (group 8, Q4_0, bf16 activations) at its contexts 50, 500 and 1500.
  * Eight slots of the Llama-3.2-1B shape (bf16 and Q4_0 + int8 head) with contexts in
    [128, 4096], four of them sharing a 512-token prefix: the few-slot GEMV's slices of
    2048 columns (K = 2048 and 8192), the wide LM head and per-slot attention splits.

Tolerances as for the other step tests: max |dlogit| <= 2e-2 * std(logits), argmax
identical where the oracle's top-2 margin exceeds 1e-2, K/V within one bf16 step of the
value plus 1e-3 of the RMS (1e-2 with bf16 activations).
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

mie = pytest.importorskip("memory_bound_decode_dequant_gb300")
from memory_bound_decode_dequant_gb300.workload import build_gpu_model  # noqa: E402

PERSISTENT, CHAIN = 0, 1
KV_SEED = 0x4B56


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)
    mie.lib()


def check_logits(got, ref, what):
    tol = 2e-2 * float(np.std(ref))
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    assert err <= tol, f"{what}: max |dlogit| {err:.3e} > {tol:.3e}"


def check_argmax(got_best, ref, what):
    top = np.sort(ref)[-2:]
    if top[1] - top[0] > 1e-2:
        assert got_best == int(np.argmax(ref)), f"{what}: argmax {got_best} vs {int(np.argmax(ref))}"


def check_kv(orc, gm, om, blocks, act_bf16):
    g = gm.kv().cpu().numpy().view(np.uint16)[blocks]
    r = om.kv()[blocks]
    gf = orc.from_bf16(g).astype(np.float64)
    rf = orc.from_bf16(r).astype(np.float64)
    rms = float(np.sqrt(np.mean(rf ** 2)))
    c = 1e-2 if act_bf16 else 1e-3
    bound = np.abs(rf) * 2.0 ** -7 + c * rms
    err = np.abs(gf - rf)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), f"K/V {worst}: gpu {gf[worst]} oracle {rf[worst]} (rms {rms:.3g})"


def prefilled_pair(orc, shape, layers, n_blocks, max_slots=1):
    """Oracle and GPU models whose KV pools hold the same seeded bf16 values."""
    max_pos = n_blocks * shape.block_size
    om = orc.Model(shape, n_kv_blocks=n_blocks, max_pos=max_pos, layers=layers)
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos, layers=layers, max_slots=max_slots)
    kv = om.kv()
    kv[...] = orc.to_bf16(synth.normal(KV_SEED, kv.size)).reshape(kv.shape)
    gm.kv().copy_(torch.from_numpy(kv.view(np.int16)).cuda())
    torch.cuda.synchronize()
    return om, gm


def run_positions(orc, shape, layers, positions, mode=PERSISTENT, n_steps=2, perm_seed=0x4254):
    bs = shape.block_size
    n_blocks = (max(positions) + n_steps + bs - 1) // bs + 2
    om, gm = prefilled_pair(orc, shape, layers, n_blocks)
    gm.set_step_mode(mode)
    bt = synth.permutation(perm_seed, n_blocks).astype(np.int32)
    btd = torch.from_numpy(bt).cuda()
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    toks = shape.tokens(len(positions), stream=7)
    written = set()
    for i, p0 in enumerate(positions):
        tok = int(toks[i])
        for pos in range(p0, p0 + n_steps):
            ref, best = om.decode_step(tok, pos, bt)
            gm.decode_step(tok, pos, btd, logits, am)
            gm.sync()
            assert gm.step_mode == mode
            what = f"{shape.name} {shape.wfmt}/{shape.head_fmt} pos {pos}"
            check_logits(logits.cpu().numpy(), ref, what)
            check_argmax(int(am.item()), ref, what)
            written.add(int(bt[pos // bs]))
            tok = best  # teacher forcing with the oracle's greedy token
    check_kv(orc, gm, om, np.array(sorted(written)), shape.act_bf16)
    gm.close()


@pytest.mark.parametrize("fmt,head,positions", [
    ("bf16", None, (150, 600, 2100, 8250)),
    ("i8", None, (150, 600, 2100)),
    ("q4_0", None, (150, 600, 2100)),
    ("q4_g128", "q4_g128", (150, 2100)),
])
def test_llama32_shape_long_context_persistent(orc, fmt, head, positions):
    run_positions(orc, synth.llama32_1b(fmt, head), 2, positions)


def test_llama32_shape_long_context_chain(orc):
    run_positions(orc, synth.llama32_1b("bf16"), 2, (150, 2100), mode=CHAIN)


@pytest.mark.parametrize("mode", [PERSISTENT, CHAIN])
def test_tinyllama_shape_contexts_50_500_1500(orc, mode):
    run_positions(orc, synth.TINYLLAMA, 2, (50, 500, 1500), mode=mode)


# ----------------------------------------------------------------------------- slots

def slot_tables(pool, contexts, bs, max_blocks, shared, prefix_blocks):
    """Block tables drawn from the context's pool: slots < shared hold the same
    prefix_blocks blocks (refcount = shared), every other block is private."""
    S = len(contexts)
    tables = np.zeros((S, max_blocks), np.int32)
    prefix = [pool.alloc() for _ in range(prefix_blocks)]
    for b in prefix:
        for _ in range(shared - 1):
            pool.incref(b)
    for s in range(S):
        for b in range((contexts[s] + 2 + bs - 1) // bs):
            tables[s, b] = prefix[b] if (s < shared and b < prefix_blocks) else pool.alloc()
    return tables, prefix


@pytest.mark.parametrize("fmt", ["bf16", "q4_0"])
def test_eight_slots_llama32_shape(orc, fmt):
    shape = synth.llama32_1b(fmt)
    bs = shape.block_size
    S, n_steps = 8, 2
    contexts = [int(c) for c in synth.uniform_int(0x534C54, S, 128, 4097)]
    contexts[:4] = [max(c, 520) for c in contexts[:4]]  # beyond the shared 512-token prefix
    max_blocks = max(contexts) // bs + 2
    n_blocks = sum((c + n_steps + bs - 1) // bs for c in contexts) + 8
    om, gm = prefilled_pair(orc, shape, 1, n_blocks, max_slots=S)
    # the pool hands out blocks in a shuffled order so tables are random physical runs
    for _ in range(n_blocks):
        assert gm.pool.alloc() >= 0
    for b in synth.permutation(0x534C, n_blocks):
        gm.pool.decref(int(b))
    tables, prefix = slot_tables(gm.pool, contexts, bs, max_blocks, shared=4, prefix_blocks=32)
    assert all(gm.pool.refcount(b) == 4 for b in prefix)
    tdev = torch.from_numpy(tables).cuda()
    logits = torch.empty((S, shape.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(S, dtype=torch.int32, device="cuda")
    cur = [int(t) for t in shape.tokens(S, stream=9)]
    pos = list(contexts)
    for step in range(n_steps):
        refs = [om.decode_step(cur[s], pos[s], tables[s]) for s in range(S)]
        gm.decode_step_slots(np.array(cur, np.int32), np.array(pos, np.int32), tdev, logits, am)
        gm.sync()
        got, best = logits.cpu().numpy(), am.cpu().numpy()
        for s in range(S):
            ref, rbest = refs[s]
            what = f"{fmt} step {step} slot {s} pos {pos[s]}"
            check_logits(got[s], ref, what)
            check_argmax(int(best[s]), ref, what)
            cur[s] = int(rbest)
            pos[s] += 1
    written = sorted({int(tables[s, p // bs]) for s in range(S) for p in range(contexts[s], pos[s])})
    check_kv(orc, gm, om, np.array(written), shape.act_bf16)
    gm.close()
