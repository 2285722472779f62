"""Pins for the allocator model (oracle/block_pool.py)."""
import copy
import json
import os

import numpy as np
import pytest

from oracle.block_pool import BlockPool, SequencePool


def test_fork_cow_example_of_the_vllm_page(golden_dir):
    with open(os.path.join(golden_dir, "block_pool_fork_cow.json")) as f:
        fx = json.load(f)
    ex = fx["expected"]
    pool = BlockPool(fx["num_blocks"], fx["block_size"])
    original = []
    for tok in fx["original_tokens"]:
        original = pool.append(original, tok).table
    branch = pool.fork(original)
    res = pool.append(branch, fx["branch_token"])
    branch = res.table
    assert pool.read(original) == ex["read_original"]
    assert pool.read(branch) == ex["read_branch"]
    assert original[-1] != branch[-1]
    assert pool.refs[original[0]] == ex["refs_original_first"]
    assert pool.refs[original[-1]] == ex["refs_original_last"]
    assert original == ex["original_table"] and branch == ex["branch_table"]
    assert list(res.cow) == ex["branch_cow_pair"]
    assert pool.free == ex["free_after"]


def test_block_counts_of_the_source_analysis_mapping_example():
    # requests of 32, 16 and 48 tokens need 2, 1 and 3 blocks of 16 (order-free property)
    pool = SequencePool(16, 16)
    ids = []
    for n in (32, 16, 48):
        sid = pool.create()
        for _ in range(n):
            pool.append(sid)
        ids.append(sid)
    assert [len(pool.tables[s]) for s in ids] == [2, 1, 3]
    used = [b for s in ids for b in pool.tables[s]]
    assert len(set(used)) == 6 and pool.num_free() == 10
    assert pool.invariants() == []


def test_slots_are_block_times_size_plus_offset():
    pool = SequencePool(4, 4)
    sid = pool.create()
    slots = [pool.append(sid).slot for _ in range(6)]
    # LIFO: first block is 3, second is 2
    assert slots == [12, 13, 14, 15, 8, 9]


def snapshot(pool):
    return copy.deepcopy((pool.pool.free, pool.pool.refs, pool.pool.data, pool.tables, pool.lens))


def test_exhaustion_leaves_state_unchanged():
    pool = SequencePool(3, 2)
    a = pool.create()
    for _ in range(5):
        pool.append(a)  # blocks 2, 1, 0; the tail holds one token; nothing is free
    b = pool.fork(a)
    snap = snapshot(pool)
    with pytest.raises(MemoryError):
        pool.append(b)  # copy-on-write of the shared tail needs a block
    assert snapshot(pool) == snap
    with pytest.raises(MemoryError):
        pool.append(a)  # a shares the tail as well
    assert snapshot(pool) == snap
    pool.release(b)
    assert pool.append(a).cow is None  # sole holder again: written in place
    full = snapshot(pool)  # a's tail is now full and the pool is empty
    with pytest.raises(MemoryError):
        pool.append(a)
    assert snapshot(pool) == full
    assert pool.invariants() == []


def test_last_sharer_writes_in_place():
    pool = SequencePool(8, 4)
    a = pool.create()
    for _ in range(6):
        pool.append(a)
    b = pool.fork(a)
    r1 = pool.append(b)
    assert r1.cow is not None  # b copies the shared tail
    r2 = pool.append(a)
    assert r2.cow is None  # a is now the only holder: in place
    assert pool.invariants() == []


@pytest.mark.parametrize("prefix,expected_copies", [(2048, 0), (2056, 63)])
def test_prefix_workload_copy_count(prefix, expected_copies):
    pool = SequencePool(1000, 16)
    parent = pool.create()
    for _ in range(prefix):
        pool.append(parent)
    seqs = [parent] + [pool.fork(parent) for _ in range(63)]
    shared = pool.tables[parent][0]
    assert pool.refcount(shared) == 64
    copies = 0
    for sid in seqs:
        copies += pool.append(sid).cow is not None
    assert copies == expected_copies
    assert pool.invariants() == []


def test_release_returns_blocks_and_keeps_shared_ones():
    pool = SequencePool(10, 2)
    a = pool.create()
    for _ in range(5):
        pool.append(a)
    b = pool.fork(a)
    pool.append(b)
    free_before = pool.num_free()
    pool.release(a)
    # a's first two blocks are still held by b; its old tail (now private to a) is freed
    assert pool.num_free() == free_before + 1
    assert pool.invariants() == []
    pool.release(b)
    assert pool.num_free() == 10
    assert pool.invariants() == []


def test_random_operations_keep_invariants():
    rng = np.random.default_rng(0)
    pool = SequencePool(64, 4, free_order=rng.permutation(64))
    live = []
    for step in range(3000):
        op = rng.integers(0, 10)
        try:
            if op == 0 or not live:
                live.append(pool.create())
            elif op == 1:
                live.append(pool.fork(live[rng.integers(len(live))]))
            elif op == 2:
                sid = live.pop(rng.integers(len(live)))
                pool.release(sid)
            else:
                pool.append(live[rng.integers(len(live))])
        except MemoryError:
            sid = live.pop(rng.integers(len(live)))
            pool.release(sid)
        assert pool.invariants() == [], step


def test_blocks_needed_hand_cases():
    pool = SequencePool(20, 4)
    a = pool.create()
    for t in range(4):  # a full tail
        pool.append(a, t)
    assert pool.blocks_needed([a], [1]) == 1 and pool.blocks_needed([a], [4]) == 1
    assert pool.blocks_needed([a], [5]) == 2
    b = pool.create()
    assert pool.blocks_needed([b], [0]) == 0 and pool.blocks_needed([b], [5]) == 2  # empty: fresh blocks
    c = pool.create()
    for t in range(6):  # one full block + a partial tail of 2
        pool.append(c, t)
    d = pool.fork(c)
    # both holders of the shared partial tail append: the first copies, the second then holds it alone
    assert pool.blocks_needed([c, d], [1, 1]) == 1
    assert pool.blocks_needed([c], [1]) == 1 and pool.blocks_needed([c], [3]) == 2
    free = pool.num_free()
    assert pool.blocks_needed([c, d, a], [2, 3, 1]) == 3
    assert pool.num_free() == free  # nothing changed


def test_blocks_needed_equals_the_blocks_the_appends_take():
    rng = np.random.default_rng(5)
    pool = SequencePool(400, 4)
    live = [pool.create()]
    for step in range(300):
        op = rng.integers(0, 6)
        if op == 0:
            live.append(pool.create())
        elif op == 1:
            live.append(pool.fork(live[rng.integers(len(live))]))
        elif op == 2 and len(live) > 1:
            pool.release(live.pop(rng.integers(len(live))))
        else:
            ids = [live[i] for i in rng.integers(0, len(live), 4)]
            counts = [int(x) for x in rng.integers(0, 7, 4)]
            need = pool.blocks_needed(ids, counts)
            if need > pool.num_free():
                continue
            free = pool.num_free()
            for sid, n in zip(ids, counts):
                for _ in range(n):
                    pool.append(sid)
            assert free - pool.num_free() == need
            assert pool.invariants() == []


def test_slots_for_positions_hand_case():
    # MiniPaged-Qwen, section 8.1: the slot of a token is its physical block times the block size plus
    # its offset in that block.  Table [7, 3] with 16-token blocks: positions 0 and 15 sit in block 7
    # (slots 112 and 127), positions 16 and 19 in block 3 (slots 48 and 51).
    from oracle import slots_for_positions

    tables = np.array([[7, 3], [5, -1]], dtype=np.int32)
    got = slots_for_positions(tables, [0, 0, 0, 0, 1, 1], [0, 15, 16, 19, 0, 9], 16)
    assert got.tolist() == [112, 127, 48, 51, 80, 89]
    assert got.dtype == np.int64


def test_slots_for_positions_agree_with_the_allocator_model():
    # The slot the allocator model's append hands back for a token, and the block and offset where
    # the model stores it, are what slots_for_positions derives from the table afterwards -- through
    # forks, copy-on-write tails and releases (the vLLM/PagedAttention page's BlockPool simulation).
    from oracle import slots_for_positions

    rng = np.random.default_rng(11)
    bs = 4
    pool = SequencePool(600, bs, free_order=rng.permutation(600))
    live = [pool.create()]
    checked = 0
    for step in range(800):
        op = rng.integers(0, 8)
        if op == 0:
            live.append(pool.create())
        elif op == 1:
            live.append(pool.fork(live[rng.integers(len(live))]))
        elif op == 2 and len(live) > 1:
            pool.release(live.pop(rng.integers(len(live))))
        elif pool.num_free() > 2:
            sid = live[rng.integers(len(live))]
            res = pool.append(sid, (sid, step))
            pos = pool.lens[sid] - 1
            tables, _ = pool.block_tables([sid], max(1, len(pool.tables[sid])))
            assert slots_for_positions(tables, [0], [pos], bs)[0] == res.slot
            checked += 1
    assert checked > 300
    # every stored token of every live sequence sits at the slot its position maps to
    width = max(len(pool.tables[s]) for s in live) or 1
    tables, lens = pool.block_tables(live, width)
    for row, sid in enumerate(live):
        tokens = pool.pool.read(pool.tables[sid])
        positions = list(range(int(lens[row])))
        slots = slots_for_positions(tables, [row] * len(positions), positions, bs)
        for pos, slot in zip(positions, slots):
            assert pool.pool.data[int(slot) // bs][int(slot) % bs] == tokens[pos]
