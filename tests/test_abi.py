"""The C ABI without a GPU: the library loads, exports every declared symbol, its host
block pool matches the oracle's, and argument checks that run before any CUDA call
return the documented status codes."""
import ctypes

import numpy as np
import pytest

import synth

mie = pytest.importorskip("memory_bound_decode_dequant_gb300")


@pytest.fixture(scope="module")
def L():
    try:
        return mie.lib()
    except RuntimeError as e:  # not built in this checkout
        pytest.skip(str(e))


def test_every_declared_function_is_exported(L):
    declared = mie.header_functions()
    assert len(declared) >= 30
    missing = [n for n in declared if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings(L):
    assert L.mie_status_string(0) == b"ok"
    assert L.mie_status_string(3) == b"out of memory"


def test_pool_matches_oracle_pool(L, orc):
    """A seeded sequence of alloc / incref / decref / copy-on-write gives the same ids,
    counts and tables in the library's pool and the oracle's (integer work: bit-exact)."""
    n = 24
    ours, ref = mie.Pool(n), orc.Pool(n, 4)
    ops = synth.uniform_int(0xB10C, 4000, 0, 4)
    picks = synth.uniform_int(0xB10D, 4000, 0, 1 << 20)
    live = []
    tables = [np.array([-1] * 4, np.int32) for _ in range(2)]
    for op, pk in zip(ops, picks):
        if op == 0:
            a, b = ours.alloc(), ref.alloc()
            assert a == b
            if a >= 0:
                live.append(a)
        elif op == 1 and live:
            i = live[pk % len(live)]
            assert (ours.incref(i) == 0) and ref.incref(i) > 0
            live.append(i)
        elif op == 2 and live:
            i = live.pop(pk % len(live))
            assert ours.decref(i) == 0
            assert ref.decref(i) >= 0
        elif op == 3 and live:
            t = tables[pk % 2]
            slot = pk % 4
            t[slot] = live[pk % len(live)]
            t2 = t.copy()
            st, blk, src, dst = ours.writable(t, slot * 16 + 3, 16)
            rblk = ref.writable(t2, slot * 16 + 3, 16)
            if st == 0:
                if dst >= 0:  # the split keeps our hold on src until the copy is queued
                    assert ours.refcount(src) >= 2
                    assert ours.decref(src) == 0
                    live.remove(src)
                    live.append(dst)
                assert blk == rblk and np.array_equal(t, t2)
            else:
                assert st == 3 and rblk == -1
        assert ours.free_count() == ref.free_count()
    for i in range(n):
        assert ours.refcount(i) == ref.refcount(i)
    assert ours.refcount(n) == -1 and ours.refcount(-1) == -1


def test_split_block_stays_held_until_released(L):
    """Copy-on-write ordering: after a split the shared block keeps this sequence's
    hold, so even when its other holder retires at once, the block is not free and
    cannot be handed out again (and overwritten) before the caller has queued its
    copy and released it."""
    p = mie.Pool(4)
    shared = p.alloc()
    p.incref(shared)                      # two sequences hold it
    table = np.array([shared], np.int32)
    st, blk, src, dst = p.writable(table, 5, 16)
    assert st == 0 and src == shared and dst == blk != shared and table[0] == blk
    assert p.decref(shared) == 0          # the other holder retires meanwhile
    assert p.refcount(shared) == 1        # ... the block is still held for the copy
    taken = [p.alloc() for _ in range(2)]
    assert shared not in taken and p.alloc() == -1
    assert p.decref(src) == 0             # copy queued: the hold is dropped
    assert p.refcount(shared) == 0 and p.alloc() == shared
    # a private block needs no split
    st, blk2, src2, dst2 = p.writable(np.array([blk], np.int32), 0, 16)
    assert (st, blk2, src2, dst2) == (0, blk, -1, -1)


def test_pool_exhaustion_is_a_status(L):
    p = mie.Pool(2)
    assert p.alloc() == 0 and p.alloc() == 1
    assert p.alloc() == -1
    assert p.decref(1) == 0 and p.alloc() == 1
    assert p.decref(5) == 1  # MIE_E_ARG for a block that is not live


def test_host_side_argument_checks(L):
    fake = ctypes.c_void_p(256)  # never dereferenced: each call fails its checks first
    assert L.mie_gemv_bf16(fake, fake, ctypes.c_void_p(512), 4, 7, None) == 2  # K % 8
    assert L.mie_gemv_i8(fake, fake, fake, ctypes.c_void_p(512), 4, 24, None) == 2  # K % 16
    assert L.mie_gemv_q4_0(fake, fake, fake, 0, 32, None) == 2
    assert L.mie_gemv_q4_0(fake, fake, fake, 4, 40000, None) == 2
    assert b"16384" in L.mie_last_error() or b"shape" in L.mie_last_error()
    assert L.mie_quantize_q4_0(None, 4, 4, fake, None) == 1
    assert L.mie_paged_attn_decode(None, fake, fake, 0, 1, fake, 1, 1, 8, 2, 32, 16, 1.0, fake, fake, 1 << 20,
                                   None) == 1
    # group size 3 and head_dim 48 are not supported
    assert L.mie_paged_attn_decode(fake, fake, fake, 4096, 4, fake, 4, 1, 6, 2, 64, 16, 1.0, fake, fake,
                                   1 << 20, None) == 2
    assert L.mie_paged_attn_decode(fake, fake, fake, 4096, 4, fake, 4, 1, 8, 2, 48, 16, 1.0, fake, fake,
                                   1 << 20, None) == 2
    # ctx_len beyond the table
    assert L.mie_paged_attn_decode(fake, fake, fake, 4096, 4, fake, 2, 33, 8, 2, 32, 16, 1.0, fake, fake,
                                   1 << 20, None) == 2
    assert L.mie_argmax(fake, 0, fake, fake, 1024, None) == 2
    # the read probe: whole aligned words only, 16- or 32-byte loads, 1..4 CTAs per SM
    assert L.mie_hbm_read_probe(None, 64, fake, 32, 2, None) == 1
    assert L.mie_hbm_read_probe(fake, 64, fake, 8, 2, None) == 1
    assert L.mie_hbm_read_probe(fake, 64, fake, 32, 5, None) == 1
    assert L.mie_hbm_read_probe(fake, 48, fake, 32, 2, None) == 2
    assert L.mie_hbm_read_probe(ctypes.c_void_p(272), 64, fake, 32, 2, None) == 2
    assert L.mie_hbm_read_probe(fake, 0, fake, 16, 2, None) == 2


def test_q4_0_packed_bytes(L):
    # nibble plane, then at a 256-byte boundary the scale plane with rows padded to 8 scales
    assert mie.mie_q4_0_packed_bytes(1, 1) == 256 + 16
    assert mie.mie_q4_0_packed_bytes(3072, 2048) == 3072 * 64 * 16 + 3072 * 64 * 2
    assert mie.mie_q4_0_packed_bytes(256, 688) == ((256 * 22 * 16 + 255) // 256) * 256 + 256 * 24 * 2


def test_config_checks_need_no_gpu(L):
    from memory_bound_decode_dequant_gb300.workload import config_for
    cfg = config_for(synth.TINY, 8, 128)
    bad = dict(cfg, n_kv_heads=3)
    with pytest.raises(mie.MieError) as e:
        mie.Model(bad, stream=0)
    assert e.value.status == 2
    with pytest.raises(mie.MieError) as e:
        mie.Model(dict(cfg, head_dim=48), stream=0)
    assert e.value.status == 2
    with pytest.raises(mie.MieError) as e:
        mie.Model(dict(cfg, max_slots=9), stream=0)
    assert e.value.status == 2


def test_binding_has_every_declared_name(L):
    """The Python binding offers each entry point of the header under its C name."""
    missing = [n for n in mie.header_functions() if not callable(getattr(mie, n, None))]
    assert not missing, missing


def test_pool_calls_by_c_name(L):
    p = mie.mie_pool_create(3)
    assert [mie.mie_pool_alloc(p) for _ in range(3)] == [0, 1, 2]
    assert mie.mie_pool_alloc(p) == -1
    mie.mie_pool_incref(p, 1)
    assert mie.mie_pool_refcount(p, 1) == 2
    table = np.array([1, -1], np.int32)
    with pytest.raises(mie.MieError) as e:  # block 1 is shared and the pool is empty
        mie.mie_pool_writable(p, table, 3, 16)
    assert e.value.status == 3 and table[0] == 1
    mie.mie_pool_decref(p, 2)
    assert mie.mie_pool_free_count(p) == 1
    blk, src, dst = mie.mie_pool_writable(p, table, 3, 16)  # copy-on-write into block 2
    assert (blk, src, dst) == (2, 1, 2) and table[0] == 2
    assert mie.mie_pool_refcount(p, 1) == 2  # still held by this sequence until the copy is queued
    mie.mie_pool_decref(p, src)
    assert mie.mie_pool_refcount(p, 1) == 1
    with pytest.raises(mie.MieError) as e:
        mie.mie_pool_decref(p, 7)
    assert e.value.status == 1
    assert mie.mie_status_string(3) == "out of memory"
    assert "mie_pool_decref" in mie.mie_last_error() or "not live" in mie.mie_last_error()
    mie.mie_pool_destroy(p)
    assert p.h is None
