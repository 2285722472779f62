"""Host-side checks of the C ABI (no GPU): exports, argument validation, and the
C++ block pool against the allocator model of the oracle."""
import copy
import json
import os
import re

import numpy as np
import pytest

import paged_kv_cache_129_gb300 as pa
from oracle.block_pool import SequencePool

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pa.build()
    return pa.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert missing == []


def test_version(lib):
    assert "sm_103a" in pa.version()


# ---- argument validation that returns before any CUDA call ---------------------------------
FAKE = 1 << 20  # an aligned, never-dereferenced address


def test_decode_rejects_bad_arguments(lib):
    ok_args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 4, 10, 0.1, 2, None, 0, 0, 0, 0, None]
    bad = list(ok_args)
    bad[0] = None  # out
    assert lib.pa_decode_ex(*bad) == 1
    bad = list(ok_args)
    bad[2] = FAKE + 2  # key cache not 16-byte aligned
    assert lib.pa_decode_ex(*bad) == 1
    bad = list(ok_args)
    bad[13] = float("nan")
    assert lib.pa_decode_ex(*bad) == 1
    bad = list(ok_args)
    bad[12] = 1 << 27  # num_blocks * H_kv * bs >= 2^31
    assert lib.pa_decode_ex(*bad) == 1
    zero = list(ok_args)
    zero[6] = 0  # no sequences: nothing to do
    assert lib.pa_decode_ex(*zero) == 0
    assert b"NULL" in lib.pa_last_error_string() or lib.pa_last_error_string() == b""


def test_write_and_copy_reject_bad_arguments(lib):
    assert lib.pa_write_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 64, 16, 4, 0, None) == 0  # no tokens
    assert lib.pa_write_kv(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 3, 2, 64, 16, 4, 0, None) == 1  # slots misaligned
    assert lib.pa_write_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 2, 64, 16, 4, 7, None) == 1  # dtype
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, 0, 2, 64, 16, 4, 0, None) == 0
    assert lib.pa_copy_blocks(None, FAKE, FAKE, 2, 2, 64, 16, 4, 0, None) == 1


def test_plan_rejects_bad_head_layout(lib):
    plan = pa.DecodePlan()
    import ctypes

    assert lib.pa_decode_make_plan(2, 6, 4, 128, 16, 8, 2, 0, 0, 0, 0, ctypes.byref(plan)) == 1
    assert b"multiple" in lib.pa_last_error_string()


# ---- block pool ------------------------------------------------------------------------------
def test_pool_fork_cow_example_of_the_vllm_page(lib, golden_dir):
    with open(os.path.join(golden_dir, "block_pool_fork_cow.json")) as f:
        fx = json.load(f)
    ex = fx["expected"]
    pool = pa.BlockPool(fx["num_blocks"], fx["block_size"])
    orig = pool.create()
    for _ in fx["original_tokens"]:
        pool.append(orig)
    branch = pool.fork(orig)
    slot, cow = pool.append(branch)
    tables, lens = pool.block_tables([orig, branch], 2)
    assert tables[0].tolist() == ex["original_table"]
    assert tables[1].tolist() == ex["branch_table"]
    assert list(cow) == ex["branch_cow_pair"]
    assert slot == ex["branch_table"][-1] * fx["block_size"] + 1
    assert pool.refcount(ex["original_table"][0]) == ex["refs_original_first"]
    assert pool.refcount(ex["original_table"][-1]) == ex["refs_original_last"]
    assert lens.tolist() == [3, 4]
    assert pool.free_list() == ex["free_after"]
    pool.check_invariants()


def pool_state(pool, ids, width):
    tables, lens = pool.block_tables(ids, width)
    refs = [pool.refcount(b) for b in range(pool.num_blocks)]
    return tables.tolist(), lens.tolist(), refs, pool.free_list()


def model_state(model, ids, width):
    tables, lens = model.block_tables(ids, width)
    refs = [model.refcount(b) for b in range(model.pool.num_blocks)]
    return tables.tolist(), lens.tolist(), refs, list(model.pool.free)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_pool_matches_allocator_model_on_random_operations(lib, seed):
    rng = np.random.default_rng(seed)
    nb, bs = 48, 4
    order = rng.permutation(nb)
    pool = pa.BlockPool(nb, bs, free_order=order)
    model = SequencePool(nb, bs, free_order=order)
    live = []  # (c++ id, model id)
    width = nb
    for step in range(1500):
        op = rng.integers(0, 12)
        if op == 0 or not live:
            live.append((pool.create(), model.create()))
        elif op == 1:
            c, m = live[rng.integers(len(live))]
            live.append((pool.fork(c), model.fork(m)))
        elif op == 2:
            c, m = live.pop(rng.integers(len(live)))
            pool.release(c)
            model.release(m)
        elif op == 3:
            k = int(rng.integers(1, len(live) + 1))
            picks = [live[i] for i in rng.choice(len(live), size=k, replace=False)]
            snap = copy.deepcopy((model.pool.free, model.pool.refs, model.pool.data, model.tables, model.lens))
            try:
                slots, pairs = pool.append_batch([c for c, _ in picks])
                exp_slots, exp_pairs = [], []
                for _, m in picks:
                    r = model.append(m)
                    exp_slots.append(r.slot)
                    if r.cow:
                        exp_pairs.append(list(r.cow))
                assert slots.tolist() == exp_slots
                assert pairs.tolist() == exp_pairs
            except pa.PoolExhausted:
                # all-or-nothing: the model must fail on one of them too; restore the model
                with pytest.raises(MemoryError):
                    for _, m in picks:
                        model.append(m)
                model.pool.free, model.pool.refs, model.pool.data, model.tables, model.lens = snap
        else:
            c, m = live[rng.integers(len(live))]
            try:
                slot, cow = pool.append(c)
            except pa.PoolExhausted:
                with pytest.raises(MemoryError):
                    model.append(m)
            else:
                r = model.append(m)
                assert slot == r.slot and cow == r.cow
        if step % 25 == 0 or step > 1400:
            pool.check_invariants()
            assert model.invariants() == []
            assert pool_state(pool, [c for c, _ in live], width) == model_state(model, [m for _, m in live], width)


def test_pool_exhaustion_leaves_state_unchanged(lib):
    pool = pa.BlockPool(3, 2)
    a = pool.create()
    for _ in range(5):
        pool.append(a)
    b = pool.fork(a)
    before = pool_state(pool, [a, b], 3)
    with pytest.raises(pa.PoolExhausted):
        pool.append(b)
    with pytest.raises(pa.PoolExhausted):
        pool.append_batch([a, b])
    assert pool_state(pool, [a, b], 3) == before
    pool.check_invariants()


def test_pool_batch_rolls_back_partial_progress(lib):
    pool = pa.BlockPool(4, 2)
    a, b = pool.create(), pool.create()
    pool.append(a)  # a: 1 token in block 3 (room for one more)
    pool.append(b)
    pool.append(b)  # b: full block 2
    before = pool_state(pool, [a, b], 4)
    free_before = pool.num_free()
    # a fits in place, b needs a block, a again needs a block, b ... -> runs out of blocks at entry 4
    with pytest.raises(pa.PoolExhausted):
        pool.append_batch([a, b, a, b, a, b, a])
    assert pool_state(pool, [a, b], 4) == before and pool.num_free() == free_before
    pool.check_invariants()


@pytest.mark.parametrize("prefix,copies", [(2048, 0), (2056, 63)])
def test_pool_prefix_workload_copy_count(lib, prefix, copies):
    pool = pa.BlockPool(1000, 16)
    parent = pool.create()
    for _ in range(prefix):
        pool.append(parent)
    seqs = [parent] + [pool.fork(parent) for _ in range(63)]
    slots, pairs = pool.append_batch(seqs)
    assert len(pairs) == copies
    assert pool.refcount(pool.block_tables([parent], 200)[0][0][0]) == 64
    pool.check_invariants()


def test_pool_unknown_sequence_and_bad_free_order(lib):
    pool = pa.BlockPool(4, 4)
    with pytest.raises(pa.PAError):
        pool.append(12345)
    with pytest.raises(pa.PAError):
        pa.BlockPool(3, 4, free_order=[0, 0, 1])
    sid = pool.create()
    for _ in range(5):
        pool.append(sid)  # two blocks
    with pytest.raises(pa.PAError):
        pool.block_tables([sid], 1)


def test_static_scratch_size_matches_the_header():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    m = re.search(r"#define PA_STATIC_SCRATCH_BYTES \((\d+)u \* 1024u \* 1024u\)", text)
    assert m and int(m.group(1)) * 1024 * 1024 == pa.STATIC_SCRATCH_BYTES
