"""Pins for the swap oracle (block copy between two pools) and the allocator model's swap.

* the byte copy: every destination block named by a pair equals the source block
  byte for byte (numpy's own indexing as the second formulation), every other
  destination byte and the whole source are unchanged, a pair with an id outside
  its own pool is skipped and reported;
* swap through the allocator model: token payloads written at the slots the model
  hands out, moved out to a second (host) pool and back with the pairs the model
  returns, read back through the new tables exactly as the model's token lists,
  and sequences that shared blocks with the moved one keep reading their tokens;
* exhaustion of the destination leaves both pools unchanged; invariants hold over
  random operation sequences that include swaps.
"""
import copy

import numpy as np
import pytest

import oracle
from oracle.block_pool import SequencePool


def test_swap_copies_blocks_between_pools():
    rng = np.random.default_rng(3)
    src_k = rng.integers(0, 2**16, (9, 2, 4, 8), dtype=np.uint16)
    src_v = rng.integers(0, 2**16, (9, 2, 4, 8), dtype=np.uint16)
    dst_k = rng.integers(0, 2**16, (5, 2, 4, 8), dtype=np.uint16)
    dst_v = rng.integers(0, 2**16, (5, 2, 4, 8), dtype=np.uint16)
    s0, d0 = (src_k.copy(), src_v.copy()), (dst_k.copy(), dst_v.copy())
    pairs = np.array([[8, 0], [3, 4], [3, 2]], np.int64)
    assert oracle.swap_blocks(dst_k, dst_v, src_k, src_v, pairs) == oracle.OK
    for s, d in pairs:
        assert dst_k[d].tobytes() == s0[0][s].tobytes()
        assert dst_v[d].tobytes() == s0[1][s].tobytes()
    np.testing.assert_array_equal(dst_k[[1, 3]], d0[0][[1, 3]])
    np.testing.assert_array_equal(dst_v[[1, 3]], d0[1][[1, 3]])
    np.testing.assert_array_equal(src_k, s0[0])
    np.testing.assert_array_equal(src_v, s0[1])


def test_swap_bad_ids_are_skipped_and_reported():
    src = np.arange(2 * 1 * 2 * 4, dtype=np.float32).reshape(2, 1, 2, 4)
    dst = np.zeros((3, 1, 2, 4), np.float32)
    dst_v = np.zeros_like(dst)
    pairs = np.array([[2, 0], [0, 3], [-1, 1], [1, 2]], np.int64)
    assert oracle.swap_blocks(dst, dst_v, src, -src, pairs) == oracle.BAD_TABLE
    np.testing.assert_array_equal(dst[:2], 0)
    np.testing.assert_array_equal(dst[2], src[1])
    np.testing.assert_array_equal(dst_v[2], -src[1])


def _payload(token, h, d):
    return np.full((1, h, d), float(token), np.float32)


class _Cached:
    """A model pool plus its K/V caches holding each token's id as payload."""

    def __init__(self, num_blocks, bs, h, d, free_order=None):
        self.pool = SequencePool(num_blocks, bs, free_order)
        self.kc = np.full((num_blocks, h, bs, d), -7.0, np.float32)
        self.vc = np.full_like(self.kc, -7.0)
        self.h, self.d = h, d

    def append(self, sid, token):
        res = self.pool.append(sid, token)
        if res.cow is not None:
            assert oracle.copy_blocks(self.kc, self.vc, np.array([res.cow])) == oracle.OK
        row = _payload(token, self.h, self.d)
        assert oracle.write_kv(row, -row, self.kc, self.vc, np.array([res.slot], np.int64)) == oracle.OK

    def read(self, sid):
        table, n, h, d = self.pool.tables[sid], self.pool.lens[sid], self.h, self.d
        k = self.kc[table].transpose(1, 0, 2, 3).reshape(h, -1, d)[:, :n]
        v = self.vc[table].transpose(1, 0, 2, 3).reshape(h, -1, d)[:, :n]
        assert (k == k[:1, :, :1]).all() and (v == -k).all()
        return [int(x) for x in k[0, :, 0]]


def _swap(src: _Cached, dst: _Cached, sid):
    new_sid, pairs = src.pool.swap_to(dst.pool, sid)
    if pairs:
        assert oracle.swap_blocks(dst.kc, dst.vc, src.kc, src.vc, np.array(pairs, np.int64)) == oracle.OK
    return new_sid, pairs


def test_swap_out_and_in_round_trip_keeps_tokens_and_sharers():
    bs, h, d = 4, 2, 3
    dev = _Cached(24, bs, h, d)
    host = _Cached(16, bs, h, d, free_order=list(range(16))[::-1])
    tok = iter(range(1000, 2000))
    parent = dev.pool.create()
    for _ in range(6):  # one full block + a shared partial tail after the fork
        dev.append(parent, next(tok))
    child = dev.pool.fork(parent)
    for _ in range(3):
        dev.append(child, next(tok))  # copy-on-write of the shared tail
    other = dev.pool.create()
    for _ in range(5):
        dev.append(other, next(tok))
    before = {s: dev.read(s) for s in (parent, child, other)}
    shared = dev.pool.tables[child][0]
    assert dev.pool.refcount(shared) == 2

    child_table = list(dev.pool.tables[child])
    hid, pairs = _swap(dev, host, child)
    assert [p[0] for p in pairs] == child_table
    assert host.pool.tables[hid] == [0, 1, 2]  # 9 tokens; LIFO from a reversed free list
    assert host.read(hid) == before[child]
    assert child not in dev.pool.tables
    assert dev.pool.refcount(shared) == 1  # the parent still holds it
    assert host.pool.refcount(0) == host.pool.refcount(1) == host.pool.refcount(2) == 1
    assert dev.read(parent) == before[parent] and dev.read(other) == before[other]
    assert dev.pool.invariants() == [] and host.pool.invariants() == []

    free_before = dev.pool.num_free()
    did, pairs_in = _swap(host, dev, hid)
    assert [p[0] for p in pairs_in] == [0, 1, 2]
    assert dev.read(did) == before[child]
    assert dev.pool.num_free() == free_before - 3 and host.pool.num_free() == 16
    # the sequence grows after coming back (its tail is private: no copy)
    dev.append(did, 4242)
    assert dev.read(did) == before[child] + [4242]
    assert dev.read(parent) == before[parent]
    assert dev.pool.invariants() == [] and host.pool.invariants() == []


def test_swap_into_a_full_pool_changes_nothing():
    dev = SequencePool(8, 2)
    host = SequencePool(2, 2)
    sid = dev.create()
    for t in range(5):
        dev.append(sid, t)
    def state():
        return [copy.deepcopy((p.tables, p.lens, p._next_id, p.pool.free, p.pool.refs, p.pool.data))
                for p in (dev, host)]

    before = state()
    with pytest.raises(MemoryError):
        dev.swap_to(host, sid)
    assert state() == before


def test_swap_empty_sequence_moves_no_block():
    dev, host = SequencePool(4, 2), SequencePool(4, 2)
    sid = dev.create()
    hid, pairs = dev.swap_to(host, sid)
    assert pairs == [] and host.tables[hid] == [] and host.lens[hid] == 0 and sid not in dev.tables


def test_swap_rejects_other_block_size():
    dev, host = SequencePool(4, 2), SequencePool(4, 4)
    with pytest.raises(ValueError):
        dev.swap_to(host, dev.create())


def test_invariants_under_random_operations_with_swaps():
    rng = np.random.default_rng(11)
    bs, h, d = 4, 1, 1
    pools = [_Cached(40, bs, h, d), _Cached(30, bs, h, d)]
    where = {}  # logical sequence -> (pool index, id)
    expect = {}
    next_seq, tok = 0, 0
    for _ in range(1500):
        op = rng.choice(["create", "append", "fork", "release", "swap"], p=[0.1, 0.55, 0.1, 0.1, 0.15])
        live = list(where)
        if op == "create" or not live:
            pi = int(rng.integers(2))
            where[next_seq] = (pi, pools[pi].pool.create())
            expect[next_seq] = []
            next_seq += 1
            continue
        s = live[int(rng.integers(len(live)))]
        pi, sid = where[s]
        try:
            if op == "append":
                pools[pi].append(sid, tok)
                expect[s].append(tok)
                tok += 1
            elif op == "fork":
                where[next_seq] = (pi, pools[pi].pool.fork(sid))
                expect[next_seq] = list(expect[s])
                next_seq += 1
            elif op == "release":
                pools[pi].pool.release(sid)
                del where[s], expect[s]
            else:
                new_sid, _ = _swap(pools[pi], pools[1 - pi], sid)
                where[s] = (1 - pi, new_sid)
        except MemoryError:
            pass
        for p in pools:
            assert p.pool.invariants() == []
    for s, (pi, sid) in where.items():
        assert pools[pi].read(sid) == expect[s]
