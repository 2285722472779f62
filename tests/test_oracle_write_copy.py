"""Pins for the byte-exact write and copy oracles.

* write: through a transpose/reshape of the cache (numpy's own route), slot s
  of kv head h is row s of the head's slot-major view, which must hold the
  written token; every other byte is unchanged; negative slots write nothing;
* write + copy + allocator: token payloads written at the slots the allocator
  model hands out, with copy-on-write pairs applied by the copy oracle, must
  read back through the block tables exactly as the allocator's own token lists
  (two independent formulations of the same state).
"""
import numpy as np
import pytest

import oracle
from oracle.block_pool import SequencePool


def slot_major(cache):
    nb, h, bs, d = cache.shape
    return cache.transpose(1, 0, 2, 3).reshape(h, nb * bs, d)


@pytest.mark.parametrize("dtype", [np.float32, np.float16, np.uint16])
def test_write_lands_in_slot_major_view(dtype):
    rng = np.random.default_rng(0)
    nb, h, bs, d, T = 6, 3, 4, 8, 9
    kc = rng.integers(0, 2**15, (nb, h, bs, d)).astype(dtype)
    vc = rng.integers(0, 2**15, (nb, h, bs, d)).astype(dtype)
    key = rng.integers(0, 2**15, (T, h, d)).astype(dtype)
    val = rng.integers(0, 2**15, (T, h, d)).astype(dtype)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[2] = -1  # padding: no write
    k0, v0 = kc.copy(), vc.copy()
    assert oracle.write_kv(key, val, kc, vc, slots) == 0
    ks, vs, ks0, vs0 = slot_major(kc), slot_major(vc), slot_major(k0), slot_major(v0)
    touched = set()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        touched.add(int(s))
        np.testing.assert_array_equal(ks[:, s], key[t])
        np.testing.assert_array_equal(vs[:, s], val[t])
    untouched = [s for s in range(nb * bs) if s not in touched]
    np.testing.assert_array_equal(ks[:, untouched], ks0[:, untouched])
    np.testing.assert_array_equal(vs[:, untouched], vs0[:, untouched])


def test_write_out_of_pool_slot_is_reported_and_skipped():
    nb, h, bs, d = 2, 1, 2, 4
    kc = np.zeros((nb, h, bs, d), np.float32)
    vc = np.zeros_like(kc)
    key = np.ones((2, h, d), np.float32)
    status = oracle.write_kv(key, key, kc, vc, np.array([nb * bs, 1], np.int64))
    assert status == oracle.BAD_SLOT
    assert kc.sum() == d  # only slot 1 written


def test_copy_blocks_copies_whole_blocks():
    rng = np.random.default_rng(1)
    kc = rng.standard_normal((8, 2, 4, 8)).astype(np.float32)
    vc = rng.standard_normal((8, 2, 4, 8)).astype(np.float32)
    k0, v0 = kc.copy(), vc.copy()
    assert oracle.copy_blocks(kc, vc, np.array([[1, 5], [2, 6]])) == 0
    np.testing.assert_array_equal(kc[5], k0[1])
    np.testing.assert_array_equal(vc[6], v0[2])
    keep = [0, 1, 2, 3, 4, 7]
    np.testing.assert_array_equal(kc[keep], k0[keep])
    np.testing.assert_array_equal(vc[keep], v0[keep])


def payload(token_id, h, d):
    """A K/V row that encodes its token id, so the cache can be read back as ids."""
    return np.full((h, d), float(token_id), np.float32)


@pytest.mark.parametrize("prefix", [6, 8])
def test_cache_reads_back_as_allocator_tokens(prefix):
    # bs 4; prefix 6 leaves a shared partial tail (copy-on-write), prefix 8 does not.
    nb, h, bs, d = 40, 2, 4, 3
    pool = SequencePool(nb, bs)
    kc = np.full((nb, h, bs, d), -1.0, np.float32)
    vc = np.full_like(kc, -1.0)
    next_id = [1000]

    def append(sid):
        tok = next_id[0]
        next_id[0] += 1
        res = pool.append(sid, tok)
        if res.cow is not None:
            assert oracle.copy_blocks(kc, vc, np.array([res.cow])) == 0
        row = payload(tok, h, d)[None]
        assert oracle.write_kv(row, -row, kc, vc, np.array([res.slot], np.int64)) == 0

    parent = pool.create()
    for _ in range(prefix):
        append(parent)
    kids = [pool.fork(parent) for _ in range(3)]
    for i, sid in enumerate([parent] + kids):
        for _ in range(i + 2):
            append(sid)
    assert pool.invariants() == []
    for sid, table in pool.tables.items():
        n = pool.lens[sid]
        rows = kc[table].transpose(1, 0, 2, 3).reshape(h, -1, d)[:, :n]
        vrows = vc[table].transpose(1, 0, 2, 3).reshape(h, -1, d)[:, :n]
        expect = np.array(pool.pool.read(table), np.float32)
        np.testing.assert_array_equal(rows[:, :, 0], np.broadcast_to(expect, (h, n)))
        np.testing.assert_array_equal(vrows[:, :, 0], -np.broadcast_to(expect, (h, n)))
