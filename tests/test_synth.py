"""The seeded input generators that both the oracle and the CUDA path draw from (CPU).

splitmix64 is pinned to its published first outputs from seed 0 and to an
implementation written here from its definition; the normal stream to Box-Muller
written out from the same integer outputs; and the counter-based properties the tests
rely on (any offset, any thread split, one row on its own) are checked bit for bit.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import synth

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def splitmix64_ref(seed: int, i: int) -> int:
    """Output i of splitmix64 from `seed` (Steele, Lea & Flood 2014): the state advances
    by the golden gamma before each output, then the 64-bit finaliser mixes it."""
    z = (seed + (i + 1) * GOLDEN) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_splitmix64_known_answers():
    # the first four outputs of splitmix64 started from state 0
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]
    assert [synth.u64(0, i) for i in range(4)] == want


@pytest.mark.parametrize("seed", [0, 1, 0x4D4945, 0xFFFFFFFFFFFFFFFF, 0x123456789ABCDEF0])
def test_splitmix64_matches_definition(seed):
    for i in (0, 1, 2, 7, 1000, 123456789, (1 << 40) + 3):
        assert synth.u64(seed, i) == splitmix64_ref(seed, i)


def test_normal_is_box_muller_of_the_integer_stream():
    seed, n = 0x5EED, 64
    got = synth.normal(seed, n, std=0.02, mean=0.5)
    for e in range(n):
        p = e >> 1
        h1, h2 = splitmix64_ref(seed, 2 * p), splitmix64_ref(seed, 2 * p + 1)
        u1 = ((h1 >> 11) + 1) * 2.0 ** -53
        u2 = (h2 >> 11) * 2.0 ** -53
        r = math.sqrt(-2.0 * math.log(u1))
        z = r * (math.sin(2 * math.pi * u2) if e & 1 else math.cos(2 * math.pi * u2))
        want = np.float32(0.5 + 0.02 * z)
        # libm and Python may differ in the last bit of a double; after rounding to
        # fp32 that is at most one fp32 step
        assert abs(int(np.float32(got[e]).view(np.int32)) - int(want.view(np.int32))) <= 1, e


def test_normal_moments():
    z = synth.normal(7, 1 << 20).astype(np.float64)
    assert abs(z.mean()) < 5 / 1024  # 5 standard errors at n = 2^20
    assert abs(z.std() - 1.0) < 5e-3
    assert abs(((z - z.mean()) ** 3).mean()) < 0.02  # symmetric
    assert abs((z ** 4).mean() - 3.0) < 0.05  # Gaussian kurtosis


def test_normal_is_counter_based():
    """Any offset and any split between threads give the same elements: the large call
    runs on several threads, the slices on one."""
    seed, n = 0xC0FFEE, 200_003
    whole = synth.normal(seed, n)
    for off, cnt in ((0, 5), (1, 4), (77_777, 1000), (n - 3, 3), (65_536, 70_000)):
        part = synth.normal(seed, cnt, offset=off)
        assert np.array_equal(part.view(np.uint32), whole[off:off + cnt].view(np.uint32))


def test_weight_rows_can_be_drawn_alone():
    shape = synth.TINY
    full = shape.weight("l1.gate")
    rows = shape.weight("l1.gate", rows=slice(100, 140))
    assert np.array_equal(rows.view(np.uint32), full[100:140].view(np.uint32))


def test_uniform_int_and_permutation():
    u = synth.uniform_int(3, 100_000, -5, 12)
    assert u.dtype == np.int32 and u.min() == -5 and u.max() == 11
    counts = np.bincount(u + 5, minlength=17)
    assert counts.min() > 0.9 * 100_000 / 17
    for n in (1, 2, 16, 1000):
        p = synth.permutation(11, n)
        assert np.array_equal(np.sort(p), np.arange(n))
    assert not np.array_equal(synth.permutation(11, 1000), np.arange(1000))
    assert np.array_equal(synth.permutation(11, 1000), synth.permutation(11, 1000))


def test_tensor_seeds_are_distinct():
    """Every weight of every workload shape draws its own stream."""
    seeds = {}
    for shape in (synth.TINY, synth.TINYLLAMA, synth.LLAMA32_1B):
        for name, _, _ in shape.tensors():
            s = shape.seed(name)
            assert s not in seeds, (shape.name, name, seeds.get(s))
            seeds[s] = (shape.name, name)
