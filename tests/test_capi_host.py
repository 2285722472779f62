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


# ---- swap between two pools (preemption) ------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1])
def test_pool_swap_matches_allocator_model(lib, seed):
    rng = np.random.default_rng(seed)
    bs, sizes = 4, (40, 24)
    orders = [rng.permutation(n) for n in sizes]
    pools = [pa.BlockPool(n, bs, free_order=o) for n, o in zip(sizes, orders)]
    models = [SequencePool(n, bs, free_order=o) for n, o in zip(sizes, orders)]
    live = []  # [pool index, c++ id, model id]
    for step in range(1200):
        op = rng.integers(0, 10)
        if op == 0 or not live:
            i = int(rng.integers(2))
            live.append([i, pools[i].create(), models[i].create()])
            continue
        k = int(rng.integers(len(live)))
        i, c, m = live[k]
        if op == 1:
            live.append([i, pools[i].fork(c), models[i].fork(m)])
        elif op == 2:
            pools[i].release(c)
            models[i].release(m)
            live.pop(k)
        elif op <= 4:
            try:
                new_c, pairs = pools[i].swap_to(pools[1 - i], c)
            except pa.PoolExhausted:
                with pytest.raises(MemoryError):
                    models[i].swap_to(models[1 - i], m)
            else:
                new_m, exp = models[i].swap_to(models[1 - i], m)
                assert pairs.tolist() == [list(p) for p in exp]
                live[k] = [1 - i, new_c, new_m]
        else:
            try:
                slot, cow = pools[i].append(c)
            except pa.PoolExhausted:
                with pytest.raises(MemoryError):
                    models[i].append(m)
            else:
                r = models[i].append(m)
                assert slot == r.slot and cow == r.cow
        if step % 50 == 0 or step > 1150:
            for j in range(2):
                pools[j].check_invariants()
                assert models[j].invariants() == []
                ids = [(c, m) for pi, c, m in live if pi == j]
                assert pool_state(pools[j], [c for c, _ in ids], sizes[j]) == \
                    model_state(models[j], [m for _, m in ids], sizes[j])


def test_pool_swap_refusals_leave_both_pools_unchanged(lib):
    dev, host = pa.BlockPool(8, 2), pa.BlockPool(2, 2)
    a = dev.create()
    for _ in range(5):
        dev.append(a)
    before = (pool_state(dev, [a], 8), pool_state(host, [], 2))
    with pytest.raises(pa.PoolExhausted):
        dev.swap_to(host, a)
    with pytest.raises(pa.PAError):
        dev.swap_to(pa.BlockPool(8, 4), a)  # other block size
    with pytest.raises(pa.PAError):
        dev.swap_to(dev, a)  # same pool
    with pytest.raises(pa.PAError):
        dev.swap_to(host, 12345)  # unknown sequence
    assert (pool_state(dev, [a], 8), pool_state(host, [], 2)) == before


def test_swap_blocks_rejects_bad_arguments(lib):
    assert lib.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 64, 16, 4, 4, 0, None) == 0  # nothing to do
    assert lib.pa_swap_blocks(None, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 16, 4, 4, 0, None) == 1
    assert lib.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 2, 2, 64, 16, 4, 4, 0, None) == 1  # pairs misaligned
    assert lib.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 16, -1, 4, 0, None) == 1  # bad pool size
    assert lib.pa_swap_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 16, 4, 4, 9, None) == 1  # dtype


# ---- block-table deltas -----------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1])
def test_pool_table_deltas_match_allocator_model(lib, seed):
    rng = np.random.default_rng(seed)
    nb, bs, rows = 160, 4, 10
    order = rng.permutation(nb)
    pool = pa.BlockPool(nb, bs, free_order=order)
    model = SequencePool(nb, bs, free_order=order)
    live = []  # (c++ id, model id)
    for step in range(600):
        op = rng.integers(0, 9)
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
            k = rng.permutation(len(live))[:rows]
            deltas, lens = pool.table_deltas([live[i][0] for i in k])
            exp, exp_lens = model.table_deltas([live[i][1] for i in k])
            assert deltas.tolist() == [list(x) for x in exp] and lens.tolist() == exp_lens
        else:
            c, m = live[rng.integers(len(live))]
            try:
                pool.append(c)
            except pa.PoolExhausted:
                with pytest.raises(MemoryError):
                    model.append(m)
            else:
                model.append(m)


def test_pool_table_deltas_refusals_change_nothing(lib):
    pool = pa.BlockPool(16, 2)
    a, b = pool.create(), pool.create()
    for _ in range(5):
        pool.append(a)
    pool.append(b)
    small = np.empty((2, 3), np.int32)
    with pytest.raises(pa.PAError):
        pool.table_deltas([a, b], out=small)  # 4 deltas do not fit in 2
    with pytest.raises(pa.PAError):
        pool.table_deltas([a, a])  # a sequence in two rows
    with pytest.raises(pa.PAError):
        pool.table_deltas([a, 999])
    deltas, lens = pool.table_deltas([a, b])  # nothing was recorded by the refused calls
    assert deltas.tolist() == [[0, 0, pool.block_tables([a], 4)[0][0, 0]], [0, 1, pool.block_tables([a], 4)[0][0, 1]],
                               [0, 2, pool.block_tables([a], 4)[0][0, 2]], [1, 0, pool.block_tables([b], 4)[0][0, 0]]]
    assert lens.tolist() == [5, 1]
    again, _ = pool.table_deltas([a, b])
    assert again.shape == (0, 3)
    pool.append(a)  # fills block 2 of a: no new entry
    pool.append(a)  # a new block
    d, _ = pool.table_deltas([a, b])
    assert d.tolist() == [[0, 3, pool.block_tables([a], 4)[0][0, 3]]]
    d, _ = pool.table_deltas([b, a])  # rows swapped: everything again
    assert [tuple(x[:2]) for x in d.tolist()] == [(0, 0), (1, 0), (1, 1), (1, 2), (1, 3)]


def test_write_layers_and_deltas_reject_bad_arguments(lib):
    import ctypes

    arr = (ctypes.c_void_p * 1)(FAKE)
    assert lib.pa_write_kv_layers(arr, arr, arr, arr, 1, FAKE, 0, 2, 64, 16, 4, 0, None) == 0  # no tokens
    assert lib.pa_write_kv_layers(arr, arr, arr, arr, 0, FAKE, 3, 2, 64, 16, 4, 0, None) == 1  # no layers
    assert lib.pa_write_kv_layers(arr, arr, arr, arr, 257, FAKE, 3, 2, 64, 16, 4, 0, None) == 1  # too many
    assert lib.pa_write_kv_layers(arr, arr, arr, arr, 1, FAKE + 4, 3, 2, 64, 16, 4, 0, None) == 1  # slots
    nul = (ctypes.c_void_p * 1)(None)
    assert lib.pa_write_kv_layers(arr, nul, arr, arr, 1, FAKE, 3, 2, 64, 16, 4, 0, None) == 1
    assert lib.pa_apply_table_deltas(FAKE, 4, 8, FAKE, 0, None) == 0
    assert lib.pa_apply_table_deltas(None, 4, 8, FAKE, 2, None) == 1
    assert lib.pa_apply_table_deltas(FAKE, 4, 8, FAKE + 2, 2, None) == 1


def test_stepper_rejects_bad_arguments(lib):
    import ctypes

    h = ctypes.c_void_p()
    assert lib.pa_stepper_create(0, None, None, None, ctypes.byref(h)) == 1 and not h.value
    assert lib.pa_stepper_create(2, None, None, None, None) == 1
    assert lib.pa_stepper_set_slot(None, 0, FAKE, FAKE, 16, FAKE, FAKE, 16) == 1
    assert lib.pa_stepper_set_call(None, 0, None) == 1
    assert lib.pa_stepper_launch(None, 0, 0, 0) == 1
    assert lib.pa_stepper_wait(None, 0) == 1
    lib.pa_stepper_destroy(None)  # a no-op


# ---- checkpoint / resume of the pool ----------------------------------------------------------
def _drive(pool, live, rng, steps):
    """Random operations; returns everything the pool answered, for comparing two pools."""
    log = []
    for _ in range(steps):
        op = int(rng.integers(0, 8))
        try:
            if op == 0 or not live:
                live.append(pool.create())
                log.append(("create", live[-1]))
            elif op == 1:
                live.append(pool.fork(live[int(rng.integers(len(live)))]))
                log.append(("fork", live[-1]))
            elif op == 2:
                pool.release(live.pop(int(rng.integers(len(live)))))
                log.append(("release",))
            elif op == 3:
                k = rng.permutation(len(live))[:6]
                d, lens = pool.table_deltas([live[i] for i in k])
                log.append(("deltas", d.tolist(), lens.tolist()))
            else:
                log.append(("append", pool.append(live[int(rng.integers(len(live)))])))
        except pa.PoolExhausted:
            log.append(("exhausted",))
    return log


def test_pool_save_load_resumes_exactly(lib):
    rng = np.random.default_rng(7)
    pool = pa.BlockPool(96, 4, free_order=rng.permutation(96))
    live = []
    _drive(pool, live, rng, 500)
    state = pool.save()
    assert len(state) == lib.pa_pool_state_size(pool._h)
    twin = pa.BlockPool.load(state)
    twin.check_invariants()
    assert twin.save() == state  # the same image
    seed = int(rng.integers(1 << 30))
    a = _drive(pool, list(live), np.random.default_rng(seed), 800)
    b = _drive(twin, list(live), np.random.default_rng(seed), 800)
    assert a == b
    assert pool.save() == twin.save()


def test_pool_load_refuses_bad_images(lib):
    pool = pa.BlockPool(8, 2)
    s = pool.create()
    for _ in range(5):
        pool.append(s)
    state = bytearray(pool.save())
    for bad in (bytes(state[:-1]), bytes(state) + b"\0", b"\0" * len(state)):
        with pytest.raises(pa.PAError):
            pa.BlockPool.load(bad)
    corrupt = bytearray(state)
    corrupt[8 * 4 + 8] ^= 0x01  # the first free-list entry
    with pytest.raises(pa.PAError):
        pa.BlockPool.load(bytes(corrupt))


def test_pool_blocks_needed_matches_allocator_model(lib):
    rng = np.random.default_rng(13)
    nb, bs = 300, 4
    order = rng.permutation(nb)
    pool = pa.BlockPool(nb, bs, free_order=order)
    model = SequencePool(nb, bs, free_order=order)
    live = [(pool.create(), model.create())]
    for step in range(400):
        op = rng.integers(0, 6)
        if op == 0:
            live.append((pool.create(), model.create()))
        elif op == 1:
            c, m = live[rng.integers(len(live))]
            live.append((pool.fork(c), model.fork(m)))
        elif op == 2 and len(live) > 1:
            c, m = live.pop(rng.integers(len(live)))
            pool.release(c)
            model.release(m)
        else:
            k = rng.integers(0, len(live), 5)
            counts = [int(x) for x in rng.integers(0, 9, 5)]
            need = pool.blocks_needed([live[i][0] for i in k], counts)
            assert need == model.blocks_needed([live[i][1] for i in k], counts)
            if need <= pool.num_free():
                for i, n in zip(k, counts):
                    for _ in range(n):
                        pool.append(live[i][0])
                        model.append(live[i][1])
    with pytest.raises(pa.PAError):
        pool.blocks_needed([123456], [1])


def test_fp8_entry_points_reject_bad_arguments(lib):
    f = float(1 / 128 ** 0.5)
    # pa_write_kv_fp8: unknown source dtype, head_dim not a multiple of 4, NULL scales; no tokens is a no-op
    assert lib.pa_write_kv_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 8, 7, None) == 1
    assert lib.pa_write_kv_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 126, 16, 8, 2, None) == 1
    assert lib.pa_write_kv_fp8(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 4, 2, 128, 16, 8, 2, None) == 1
    assert lib.pa_write_kv_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 128, 16, 8, 2, None) == 0
    # pa_decode_fp8: NULL scales, misaligned query, f32 queries (no FP8 kernel for them)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 4, 10, f, 2, FAKE, 1 << 20, None]
    bad = list(args)
    bad[4] = None
    assert lib.pa_decode_fp8(*bad) == 1
    bad = list(args)
    bad[1] = FAKE + 4
    assert lib.pa_decode_fp8(*bad) == 1
    bad = list(args)
    bad[16] = 0  # PA_F32
    assert lib.pa_decode_fp8(*bad) == 2
    zero = list(args)
    zero[8] = 0  # no sequences
    assert lib.pa_decode_fp8(*zero) == 0
    # pa_decode_fp8_append: NULL or misaligned new rows, NULL scales, f32 queries; no sequences is a no-op
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 4, 10, f, 2, FAKE, 1 << 20,
            None]
    for i, v in ((2, None), (3, None), (3, FAKE + 8), (6, None), (7, None)):
        bad = list(args)
        bad[i] = v
        assert lib.pa_decode_fp8_append(*bad) == 1, i
    bad = list(args)
    bad[18] = 0  # PA_F32
    assert lib.pa_decode_fp8_append(*bad) == 2
    zero = list(args)
    zero[10] = 0
    assert lib.pa_decode_fp8_append(*zero) == 0
