"""The few-slot decode step on the GPU against the oracle.

The oracle defines the batched step as independent single-slot steps, one per slot,
each through its own block table of the shared pool.  Here four slots of a
tiny-shaped decoder (bf16, int8 or Q4_0 weights) are prefilled by single-slot steps, slots 0
and 1 sharing a two-block prefix (refcount 2 in the host pool), then advanced together
by batched steps, teacher-forced with the oracle's greedy tokens.  Tolerances as for
the single-slot step: max |dlogit| <= 2e-2 * std(logits), argmax identical where the
oracle's top-2 margin exceeds 1e-2, K/V within one bf16 step plus 1e-3 of the RMS.
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


def check_slot(got, ref, what):
    tol = 2e-2 * float(np.std(ref))
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    assert err <= tol, f"{what}: max |dlogit| {err:.3e} > {tol:.3e}"


def tables_with_prefix(pool, lengths, bs, max_blocks, shared=2, prefix_blocks=2):
    """Block tables for every slot: slots < shared share the first prefix_blocks blocks."""
    S = len(lengths)
    tables = np.zeros((S, max_blocks), np.int32)
    prefix = [pool.alloc() for _ in range(prefix_blocks)]
    for s in range(S):
        nb = (lengths[s] + bs - 1) // bs
        for b in range(nb):
            if s < shared and b < prefix_blocks:
                tables[s, b] = prefix[b]
                if s > 0:
                    pool.incref(prefix[b])
            else:
                tables[s, b] = pool.alloc()
    return tables, prefix


def run_slots(orc, shape, n_slots, max_slots, prompts, n_gen, compare_kv=True, n_blocks=64, max_pos=128):
    bs = shape.block_size
    lengths = [p + n_gen for p in prompts]
    max_blocks = max((n + bs - 1) // bs for n in lengths) + 1
    pool = mie.Pool(n_blocks)
    tables, prefix = tables_with_prefix(pool, lengths, bs, max_blocks)
    assert all(pool.refcount(b) == 2 for b in prefix)
    shared_len = 2 * bs
    toks = [list(prompt_tokens(shape, prompts[s], stream=s)) for s in range(n_slots)]
    toks[1][:shared_len] = toks[0][:shared_len]  # the shared prefix holds the same tokens

    om = orc.Model(shape, n_kv_blocks=n_blocks, max_pos=max_pos)
    gm = build_gpu_model(shape, n_kv_blocks=n_blocks, max_pos=max_pos, max_slots=max_slots)
    tdev = torch.from_numpy(tables).cuda()
    logits1 = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    am1 = torch.empty(1, dtype=torch.int32, device="cuda")
    # prefill each slot with single-slot steps up to its last prompt token; slot 1 starts
    # after the shared prefix, which slot 0 wrote
    for s in range(n_slots):
        for pos in range(shared_len if s == 1 else 0, prompts[s] - 1):
            om.decode_step(int(toks[s][pos]), pos, tables[s])
            gm.decode_step(int(toks[s][pos]), pos, tdev[s], logits1, am1)
    gm.sync()

    logits = torch.empty((n_slots, shape.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(n_slots, dtype=torch.int32, device="cuda")
    cur = [int(toks[s][prompts[s] - 1]) for s in range(n_slots)]
    pos = [prompts[s] - 1 for s in range(n_slots)]
    for step in range(n_gen):
        refs = [om.decode_step(cur[s], pos[s], tables[s]) for s in range(n_slots)]
        gm.decode_step_slots(np.array(cur, np.int32), np.array(pos, np.int32), tdev[:n_slots], logits, am)
        gm.sync()
        got = logits.cpu().numpy()
        best = am.cpu().numpy()
        for s in range(n_slots):
            ref, rbest = refs[s]
            check_slot(got[s], ref, f"step {step} slot {s}")
            top = np.sort(ref)[-2:]
            if top[1] - top[0] > 1e-2:
                assert int(best[s]) == int(np.argmax(ref)), f"step {step} slot {s}: argmax"
            cur[s] = int(rbest)
            pos[s] += 1
    if compare_kv:
        used = np.unique(np.concatenate([tables[s, : (lengths[s] + bs - 1) // bs] for s in range(n_slots)]))
        g = gm.kv().cpu().numpy().view(np.uint16)[used]
        r = om.kv()[used]
        gf = orc.from_bf16(g).astype(np.float64)
        rf = orc.from_bf16(r).astype(np.float64)
        rms = float(np.sqrt(np.mean(rf[rf != 0] ** 2)))
        bound = np.abs(rf) * 2.0 ** -7 + 1e-3 * rms
        err = np.abs(gf - rf)
        worst = np.unravel_index(np.argmax(err / bound), err.shape)
        assert np.all(err <= bound), f"K/V {worst}: gpu {gf[worst]} oracle {rf[worst]}"
    # retiring a slot releases its blocks; the shared prefix survives until both are gone
    for b in tables[1, : (lengths[1] + bs - 1) // bs]:
        pool.decref(int(b))
    assert all(pool.refcount(b) == 1 for b in prefix)
    return gm


@pytest.mark.parametrize("fmt", ["bf16", "i8", "q4_0", "q4_g64", "q4_g128"])
def test_slots_match_single_slot_oracle(orc, fmt):
    shape = replace(synth.TINY, wfmt=fmt, head_fmt=fmt)
    run_slots(orc, shape, n_slots=4, max_slots=4, prompts=[40, 37, 21, 50], n_gen=6)


def test_slots_long_context_loops_over_splits(orc):
    """A slot whose context needs more 256-token splits than the few-slot attention grid
    has CTAs per (KV head, slot) (16): each CTA then loops over several splits."""
    shape = replace(synth.TINY, wfmt="bf16", head_fmt="bf16")
    run_slots(orc, shape, n_slots=2, max_slots=2, prompts=[4200, 300], n_gen=2, compare_kv=False,
              n_blocks=300, max_pos=4224)


@pytest.mark.parametrize("fmt", ["bf16", "q4_0"])
def test_eight_slots_the_maximum(orc, fmt):
    """All eight slots (the largest batch a context takes) with uneven contexts."""
    shape = replace(synth.TINY, wfmt=fmt, head_fmt=fmt)
    run_slots(orc, shape, n_slots=8, max_slots=8, prompts=[40, 37, 21, 50, 18, 33, 45, 26], n_gen=3)


def test_fewer_slots_than_the_context_holds(orc):
    """n_slots < max_slots: the unused slots' lanes of every tile carry zeros."""
    shape = replace(synth.TINY, wfmt="bf16", head_fmt="bf16")
    run_slots(orc, shape, n_slots=3, max_slots=8, prompts=[35, 33, 18], n_gen=4, compare_kv=False)


def test_slots_reject_bad_inputs_and_unbuilt_formats():
    shape = replace(synth.TINY, wfmt="bf16", head_fmt="bf16")
    gm = build_gpu_model(shape, n_kv_blocks=8, max_pos=64, max_slots=2)
    tdev = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    logits = torch.empty((2, shape.vocab), dtype=torch.float32, device="cuda")
    with pytest.raises(mie.MieError) as e:  # more slots than the context was built for
        gm.decode_step_slots(np.array([1, 2, 3], np.int32), np.array([0, 0, 0], np.int32),
                             torch.zeros((3, 4), dtype=torch.int32, device="cuda"), logits)
    assert e.value.status == 1
    with pytest.raises(mie.MieError) as e:  # token outside the vocabulary
        gm.decode_step_slots(np.array([1, shape.vocab], np.int32), np.array([0, 0], np.int32), tdev, logits)
    assert e.value.status == 1
    with pytest.raises(mie.MieError) as e:  # position beyond the table
        gm.decode_step_slots(np.array([1, 2], np.int32), np.array([0, 4 * 16], np.int32), tdev, logits)
    assert e.value.status == 1
    gq = build_gpu_model(synth.TINY, n_kv_blocks=8, max_pos=64, max_slots=2)  # Q4_0 layers
    tq = torch.tensor([[0, 1, 2, 3], [4, 5, 6, 7]], dtype=torch.int32, device="cuda")
    gq.decode_step_slots(np.array([1, 2], np.int32), np.array([0, 0], np.int32), tq, logits)
    gq.sync()
