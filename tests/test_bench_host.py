"""Host logic of bench.py on CPU: byte accounting, per-rank seeds, and the
max/sum over ranks with a world-size-2 gloo process group."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_decode_bytes_counts_valid_tokens_q_out_tables_lengths():
    lens = [1, 16, 17]
    got = bench.decode_bytes(lens, num_heads=8, num_kv_heads=2, head_dim=64, elem_bytes=2, block_size=16)
    kv = 2 * sum(lens) * 2 * 64 * 2
    qo = 2 * 3 * 8 * 64 * 2
    tables = 4 * (1 + 1 + 2)
    assert got == kv + qo + tables + 4 * 3


def test_kv_size_formula_matches_the_pages_worked_numbers():
    # M_KV = 2 L b H_kv d_h sum T: LLaMA-7B (32 layers, 32 kv heads, d 128, fp16) at 4096 tokens ~ 2.15 GB,
    # and 32 layers x hidden 4096 x batch 8 x seq 2048 fp16 ~ 8.6 GB.
    per_layer = bench.decode_bytes([4096], 32, 32, 128, 2, 16) - 2 * 32 * 128 * 2 - 4 * 256 - 4
    assert abs(32 * per_layer / 1e9 - 2.147) < 0.01
    per_layer8 = bench.decode_bytes([2048] * 8, 32, 32, 128, 2, 16) - 2 * 8 * 32 * 128 * 2 - 4 * 8 * 128 - 32
    assert abs(32 * per_layer8 / 1e9 - 8.59) < 0.01


def test_rank_seeds_differ_and_rank0_keeps_the_base_seed():
    seeds = {bench.rank_seed(7, r) for r in range(8)}
    assert len(seeds) == 8 and bench.rank_seed(7, 0) == 7


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + rank, world)
        s = bench.sum_over_ranks(1.5 * (rank + 1), world)
        bench.barrier(world)
        out[rank] = (t, s)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as sck:
        sck.bind(("127.0.0.1", 0))
        return sck.getsockname()[1]


def test_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (11.0, 4.5)


@pytest.mark.parametrize("workload,copies", [("prefix_cow", 0), ("prefix_cow_2056", 63)])
def test_prefix_setup_through_the_block_pool(workload, copies):
    inp, tables, lens, slots, n_cow, unique = bench.prefix_batch(workload, 0)
    assert n_cow == copies
    bs = inp.block_size
    # the step's new token sits at position L - 1 of every sequence
    derived = tables[np.arange(len(lens)), (lens - 1) // bs].astype(np.int64) * bs + (lens - 1) % bs
    assert np.array_equal(slots, derived)
    # the shared prefix blocks are the same physical blocks in every table
    shared = (2056 if copies else 2048) // bs
    assert (tables[:, :shared] == tables[0, :shared]).all()
    # distinct pages are far fewer than the pages all sequences read
    touched = bench.pages_touched_bytes(lens, inp.num_kv_heads, inp.head_dim, 2, bs)
    assert unique < touched / 8


def test_verify_setup_slots_are_the_last_q_len_positions():
    from paged_kv_cache_129_gb300 import workloads as wl

    inp = wl.make_decode_inputs("v", context_lens=[5, 16, 40, 33], num_heads=8, num_kv_heads=2, head_dim=64,
                                block_size=16, dtype="bf16", pool_slack=0.5, seed=1, with_new_token=True, q_len=4)
    tables, lens, slots = bench.pool_tables(inp)
    assert slots.shape == (4 * 4,)
    bs = 16
    for b in range(4):
        for t in range(4):
            pos = int(lens[b]) - 4 + t
            assert slots[b * 4 + t] == int(tables[b, pos // bs]) * bs + pos % bs


def test_swap_plan_moves_each_group_out_and_back():
    import paged_kv_cache_129_gb300 as pa

    pa.build()
    plan, host_blocks, pool_s, lens = bench.swap_plan(seed=3, steps=4, num_blocks=2100, num_seqs=8, group=3,
                                                      block_size=16)
    need = (lens + 15) // 16
    assert host_blocks == int(np.sort(need)[-3:].sum())  # room for the three longest sequences
    for k, (out_p, ho, in_p, hi) in enumerate(plan):
        out_seqs = [(k * 3 + j) % 8 for j in range(3)]
        assert len(out_p) == int(need[out_seqs].sum()) and ho == k % 2
        assert len(set(out_p[:, 0].tolist())) == len(out_p) and len(set(out_p[:, 1].tolist())) == len(out_p)
        assert (out_p[:, 0] < 2100).all() and (out_p[:, 1] < host_blocks).all()
        if k == 0:
            assert len(in_p) == 0
            continue
        prev_out, prev_ho = plan[k - 1][0], plan[k - 1][1]
        # the previous group comes back from the host pool it went to
        assert hi == prev_ho and sorted(in_p[:, 0].tolist()) == sorted(prev_out[:, 1].tolist())
        # the two copies of a step touch disjoint blocks: device side and host side
        assert set(in_p[:, 1].tolist()).isdisjoint(out_p[:, 0].tolist())
        assert hi != ho
    assert pool_s >= 0


def test_reference_arm_tables_come_from_the_allocator_model_and_match_the_product_pool():
    # The reference arm builds tables, slots, copy-on-write pairs and swap pairs with the oracle's
    # allocator model; with the same free order they equal the product pool's, so both arms time the
    # same workload.
    import paged_kv_cache_129_gb300 as pa
    from paged_kv_cache_129_gb300 import workloads as wl

    pa.build()
    inp = wl.make_decode_inputs("v", context_lens=[5, 16, 40, 33, 2], num_heads=8, num_kv_heads=2, head_dim=64,
                                block_size=16, dtype="bf16", pool_slack=0.5, seed=2, with_new_token=True, q_len=2)
    for got, want in zip(bench.pool_tables(inp, model=True), bench.pool_tables(inp)):
        assert np.array_equal(got, want)
    for workload in ("prefix_cow", "prefix_cow_2056"):
        m = bench.prefix_batch(workload, 0, model=True)
        p = bench.prefix_batch(workload, 0)
        for i in (1, 2, 3):
            assert np.array_equal(m[i], p[i])
        assert m[4] == p[4] and m[5] == p[5]
        assert np.array_equal(m[0].key_cache, p[0].key_cache) and np.array_equal(m[0].value_cache, p[0].value_cache)
    mp_, mh, _, ml = bench.swap_plan(seed=3, steps=3, num_blocks=2100, num_seqs=8, group=3, model=True)
    pp, ph, _, pl = bench.swap_plan(seed=3, steps=3, num_blocks=2100, num_seqs=8, group=3)
    assert mh == ph and np.array_equal(ml, pl)
    for a, b in zip(mp_, pp):
        assert np.array_equal(a[0], b[0]) and a[1] == b[1] and np.array_equal(a[2], b[2]) and a[3] == b[3]


def test_reference_arm_setup_maps_no_product_library():
    # Built with the allocator model, the reference arm's inputs need nothing from the CUDA library.
    import subprocess
    import sys

    code = ("import bench, numpy as np\n"
            "from paged_kv_cache_129_gb300 import workloads as wl\n"
            "inp = wl.make_decode_inputs('v', context_lens=[5, 40], num_heads=4, num_kv_heads=2, head_dim=64,"
            " block_size=16, dtype='bf16', pool_slack=0.5, seed=2, with_new_token=True)\n"
            "bench.pool_tables(inp, model=True)\n"
            "bench.prefix_batch('prefix_cow_2056', 0, model=True)\n"
            "bench.swap_plan(seed=3, steps=2, num_blocks=2100, num_seqs=8, group=3, model=True)\n"
            "maps = open('/proc/self/maps').read()\n"
            "assert 'libpagedkv' not in maps, 'product library mapped'\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.run([sys.executable, "-c", code], cwd=root, check=True, timeout=300)


def test_default_line_side_records_and_schedule_names():
    # every side record of the default line is a known workload, and every plan schedule the library
    # reports (0 grid, 1 lean, 2 row split) has a name in the line
    assert set(bench.SIDE_WORKLOADS) <= set(bench.WORKLOAD_DESCRIPTIONS)
    assert "qwen_gqa" not in bench.SIDE_WORKLOADS
    assert set(bench.SCHEDULE_NAMES) == {0, 1, 2}
