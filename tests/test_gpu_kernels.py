"""GPU parity of the three kernels against the oracle on small, ragged and edge cases.

Decode: fp32 max abs error <= 1e-5; bf16/fp16 |err| <= 2e-2 + 1e-2 |ref|.
Write and copy: bit-exact, and untouched bytes unchanged.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from paged_kv_cache_129_gb300 import workloads as wl
from helpers import assert_decode_close, slots_of, to_device, to_f64, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    pa.library()
    yield
    pa.check_error()


def upload(inp):
    return dict(
        q=to_device(inp.q, inp.dtype),
        kc=to_device(inp.key_cache, inp.dtype),
        vc=to_device(inp.value_cache, inp.dtype),
        bt=torch.from_numpy(inp.block_tables).cuda(),
        lens=torch.from_numpy(inp.context_lens).cuda(),
    )


def gpu_decode(inp, dev=None, partition_pages=0, kernel="auto", max_context_len=0):
    dev = dev or upload(inp)
    ws = None
    if partition_pages >= 0:
        plan = pa.decode_plan(inp.num_seqs, inp.num_heads, inp.num_kv_heads, inp.head_dim, inp.block_size,
                              inp.max_blocks_per_seq, dev["q"].dtype, max_context_len=max_context_len,
                              partition_pages=partition_pages, kernel=kernel)
        if plan.workspace_bytes:
            ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    out = pa.decode(dev["q"], dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws,
                    partition_pages=partition_pages, kernel=kernel, max_context_len=max_context_len)
    torch.cuda.synchronize()
    return out


def case(dtype, d, bs, hq, hkv, lens, seed=0, slack=0.5):
    return wl.make_decode_inputs(f"case_{dtype}", context_lens=list(lens), num_heads=hq, num_kv_heads=hkv,
                                 head_dim=d, block_size=bs, dtype=dtype, pool_slack=slack, seed=seed)


# ---- decode ----------------------------------------------------------------------------------
@pytest.mark.parametrize("partition_pages", [0, 1, 2, -1])
def test_tiny_workload(partition_pages):
    inp = wl.tiny()
    ref = oracle.decode_inputs(inp)
    got = to_f64(gpu_decode(inp, partition_pages=partition_pages))
    assert_decode_close(got, ref, "f32")
    pa.check_error()


RAGGED = (0, 1, 15, 16, 17, 31, 32, 33, 100, 257, 700)

CASES = [
    # dtype, d, bs, hq, hkv, kernel
    ("bf16", 128, 16, 28, 4, "mma"),
    ("bf16", 128, 16, 32, 8, "mma"),
    ("bf16", 128, 16, 8, 8, "mma"),
    ("bf16", 128, 32, 28, 4, "mma"),
    ("bf16", 64, 16, 12, 2, "mma"),
    ("bf16", 256, 16, 8, 2, "mma"),
    ("bf16", 256, 32, 4, 4, "mma"),
    ("f16", 128, 16, 32, 32, "mma"),
    ("f16", 128, 32, 32, 32, "mma"),
    ("f16", 64, 32, 16, 2, "mma"),  # g = 8
    ("f16", 128, 16, 32, 2, "mma"),  # g = 16: two head chunks
    ("bf16", 128, 16, 6, 2, "mma"),  # g = 3
    ("bf16", 128, 16, 28, 4, "simt"),
    ("bf16", 128, 32, 32, 8, "simt"),
    ("f16", 128, 16, 32, 32, "simt"),
    ("f16", 128, 16, 24, 2, "simt"),  # g = 12: two chunks of 8
    ("f32", 64, 16, 4, 2, "simt"),
    ("f32", 128, 16, 28, 4, "simt"),
    ("f32", 128, 32, 8, 8, "simt"),
    ("f32", 64, 32, 6, 3, "simt"),
]


@pytest.mark.parametrize("dtype,d,bs,hq,hkv,kernel", CASES)
@pytest.mark.parametrize("partition_pages", [0, 3, -1])
def test_decode_matches_oracle(dtype, d, bs, hq, hkv, kernel, partition_pages):
    inp = case(dtype, d, bs, hq, hkv, RAGGED, seed=zlib.crc32(f"{dtype}{d}{bs}{hq}{hkv}".encode()) % 1000)
    ref = oracle.decode_inputs(inp)
    got = to_f64(gpu_decode(inp, partition_pages=partition_pages, kernel=kernel))
    assert_decode_close(got, ref, dtype)
    pa.check_error()


@pytest.mark.parametrize("partition_pages", [1, 2, 5, 64])
def test_every_partition_size_agrees(partition_pages):
    # split-KV with any partition size equals the single pass up to rounding
    inp = case("bf16", 128, 16, 28, 4, (5, 16, 80, 333, 1024), seed=21)
    ref = oracle.decode_inputs(inp)
    single = to_f64(gpu_decode(inp, partition_pages=-1))
    split = to_f64(gpu_decode(inp, partition_pages=partition_pages))
    assert_decode_close(split, ref, "bf16")
    assert np.abs(split - single).max() < 2e-2


def test_masked_tail_and_unused_blocks_may_hold_nan():
    for dtype, kernel in (("bf16", "mma"), ("f16", "simt"), ("f32", "simt")):
        inp = case(dtype, 128, 16, 8, 2, (3, 17, 31, 50), seed=3, slack=1.0)
        ref = oracle.decode_inputs(inp)
        kc, vc = inp.key_cache.copy(), inp.value_cache.copy()
        nan = {"f32": np.float32(np.nan), "f16": np.float16(np.nan), "bf16": np.uint16(0x7FC0)}[dtype]
        used = set()
        for b, L in enumerate(inp.context_lens):
            nblk = -(-int(L) // inp.block_size)
            used.update(int(x) for x in inp.block_tables[b, :nblk])
            last = inp.block_tables[b, nblk - 1]
            kc[last, :, int(L) - (nblk - 1) * inp.block_size:, :] = nan
            vc[last, :, int(L) - (nblk - 1) * inp.block_size:, :] = nan
        for blk in set(range(inp.num_blocks)) - used:
            kc[blk] = nan
            vc[blk] = nan
        inp.key_cache, inp.value_cache = kc, vc
        got = to_f64(gpu_decode(inp, kernel=kernel, partition_pages=1))
        assert_decode_close(got, ref, dtype)


def test_zero_length_contexts_give_zero_rows():
    inp = case("bf16", 128, 16, 8, 2, (0, 20, 0), seed=4)
    got = to_f64(gpu_decode(inp, partition_pages=1))
    assert (got[0] == 0).all() and (got[2] == 0).all()
    assert_decode_close(got, oracle.decode_inputs(inp), "bf16")


def test_output_is_deterministic():
    inp = case("bf16", 128, 16, 28, 4, (400, 1000, 77), seed=5)
    a = gpu_decode(inp, partition_pages=4).clone()
    b = gpu_decode(inp, partition_pages=4)
    assert torch.equal(a, b)


def test_runs_on_a_side_stream():
    inp = case("f16", 128, 16, 32, 32, (64, 129), seed=6)
    dev = upload(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = pa.decode(dev["q"], dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale)
    s.synchronize()
    assert_decode_close(to_f64(out), oracle.decode_inputs(inp), "f16")


def test_bad_table_entry_is_flagged_not_faulted():
    inp = case("bf16", 128, 16, 8, 2, (40, 40), seed=7)
    dev = upload(inp)
    dev["bt"][1, 1] = inp.num_blocks + 5  # outside the pool
    pa.decode(dev["q"], dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale)
    with pytest.raises(pa.PAError) as e:
        pa.check_error()
    assert e.value.status == 5
    pa.check_error()  # cleared


def test_context_longer_than_its_table_is_flagged():
    inp = case("bf16", 128, 16, 8, 2, (40, 40), seed=8)
    dev = upload(inp)
    dev["lens"][0] = inp.max_blocks_per_seq * inp.block_size + 1
    pa.decode(dev["q"], dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale)
    with pytest.raises(pa.PAError) as e:
        pa.check_error()
    assert e.value.status == 7


def test_scale_is_applied():
    inp = case("f32", 64, 16, 4, 2, (30, 45), seed=9)
    inp.scale = 0.37
    assert_decode_close(to_f64(gpu_decode(inp)), oracle.decode_inputs(inp), "f32")


# ---- write and copy --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 36])
def test_write_kv_is_bit_exact(dtype, d):
    rng = np.random.default_rng(d)
    nb, hkv, bs, T = 20, 3, 16, 37
    kc = wl.cast_from_f32(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
    vc = wl.cast_from_f32(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
    key = wl.cast_from_f32(rng.standard_normal((T, hkv, d)).astype(np.float32), dtype)
    val = wl.cast_from_f32(rng.standard_normal((T, hkv, d)).astype(np.float32), dtype)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[[3, 9]] = -1
    dk, dv = to_device(kc, dtype), to_device(vc, dtype)
    pa.write_kv(to_device(key, dtype), to_device(val, dtype), dk, dv, torch.from_numpy(slots).cuda())
    ek, ev = kc.copy(), vc.copy()
    assert oracle.write_kv(key, val, ek, ev, slots) == 0
    assert np.array_equal(to_host(dk, dtype).view(np.uint8), ek.view(np.uint8))
    assert np.array_equal(to_host(dv, dtype).view(np.uint8), ev.view(np.uint8))
    pa.check_error()


def test_write_kv_flags_slot_past_the_pool():
    nb, hkv, bs, d = 4, 2, 16, 64
    kc = torch.zeros(nb, hkv, bs, d, device="cuda")
    vc = torch.zeros_like(kc)
    key = torch.ones(2, hkv, d, device="cuda")
    pa.write_kv(key, key, kc, vc, torch.tensor([nb * bs, 5], device="cuda"))
    with pytest.raises(pa.PAError) as e:
        pa.check_error()
    assert e.value.status == 6
    assert kc.sum().item() == hkv * d  # the valid token landed


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_copy_blocks_is_bit_exact(dtype):
    rng = np.random.default_rng(11)
    nb, hkv, bs, d = 30, 4, 16, 128
    kc = wl.cast_from_f32(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
    vc = wl.cast_from_f32(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
    pairs = np.array([[3, 10], [4, 11], [27, 0], [5, 29]], dtype=np.int64)
    dk, dv = to_device(kc, dtype), to_device(vc, dtype)
    pa.copy_blocks(dk, dv, torch.from_numpy(pairs).cuda())
    assert oracle.copy_blocks(kc, vc, pairs) == 0
    assert np.array_equal(to_host(dk, dtype).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(to_host(dv, dtype).view(np.uint8), vc.view(np.uint8))
    pa.check_error()


def test_copy_blocks_flags_bad_ids():
    kc = torch.zeros(4, 1, 16, 64, device="cuda")
    vc = torch.zeros_like(kc)
    pa.copy_blocks(kc, vc, torch.tensor([[0, 9]], device="cuda"))
    with pytest.raises(pa.PAError) as e:
        pa.check_error()
    assert e.value.status == 5


def test_write_then_decode_sees_the_new_token():
    inp = case("bf16", 128, 16, 28, 4, (100, 513, 2048), seed=12)
    rng = np.random.default_rng(3)
    hkv, d = inp.num_kv_heads, inp.head_dim
    newk = wl.cast_from_f32(rng.standard_normal((3, hkv, d)).astype(np.float32), "bf16")
    newv = wl.cast_from_f32(rng.standard_normal((3, hkv, d)).astype(np.float32), "bf16")
    pos = inp.context_lens.astype(np.int64) - 1
    slots = slots_of(inp.block_tables, range(3), pos, inp.block_size)
    dev = upload(inp)
    pa.write_kv(to_device(newk, "bf16"), to_device(newv, "bf16"), dev["kc"], dev["vc"],
                torch.from_numpy(slots).cuda())
    got = to_f64(gpu_decode(inp, dev=dev))
    assert oracle.write_kv(newk, newv, inp.key_cache, inp.value_cache, slots) == 0
    assert_decode_close(got, oracle.decode_inputs(inp), "bf16")


# ---- lean (stream-K) schedule ------------------------------------------------------------------
LEAN_LENS = [
    (1,),
    (0, 0, 0),
    (5, 0, 2000, 0, 17),
    tuple(range(0, 700, 7)),
    (4096,) * 3 + (1,) * 40,
]


@pytest.mark.parametrize("lens", LEAN_LENS, ids=["one", "all_empty", "mixed", "ramp100", "skewed"])
@pytest.mark.parametrize("dtype,kernel,hq,hkv", [("bf16", "mma", 28, 4), ("f16", "mma", 32, 2),
                                                  ("f16", "simt", 8, 2), ("f32", "simt", 4, 2)])
def test_lean_schedule_matches_oracle(lens, dtype, kernel, hq, hkv):
    inp = case(dtype, 128, 16, hq, hkv, lens, seed=len(lens) + hq)
    plan = pa.decode_plan(inp.num_seqs, hq, hkv, 128, 16, inp.max_blocks_per_seq, TORCH[dtype], kernel=kernel)
    assert plan.schedule == 1
    got = to_f64(gpu_decode(inp, kernel=kernel))
    assert_decode_close(got, oracle.decode_inputs(inp), dtype)
    pa.check_error()


def test_lean_workspace_is_reusable_across_calls():
    # the per-unit arrival counters must be back at zero after every call
    plan = pa.decode_plan(64, 28, 4, 128, 16, 300, torch.bfloat16)
    grid = pa.decode_plan(64, 28, 4, 128, 16, 300, torch.bfloat16, partition_pages=3)
    ws = torch.zeros(max(plan.workspace_bytes, grid.workspace_bytes), dtype=torch.uint8, device="cuda")
    for seed, lens in ((1, (300 * 16, 17, 4000, 1)), (2, (1000,) * 9), (3, tuple(range(1, 4800, 97)))):
        inp = case("bf16", 128, 16, 28, 4, lens, seed=seed)
        dev = upload(inp)
        ref = oracle.decode_inputs(inp)
        for pp in (0, 3, 0):  # lean, partitioned grid, lean again on the same workspace
            out = pa.decode(dev["q"], dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws,
                            partition_pages=pp)
            torch.cuda.synchronize()
            assert_decode_close(to_f64(out), ref, "bf16")
    pa.check_error()


def test_many_sequences_fall_back_to_the_partitioned_grid():
    inp = case("bf16", 128, 16, 4, 4, (1, 3) * 2100, seed=30)
    plan = pa.decode_plan(inp.num_seqs, 4, 4, 128, 16, inp.max_blocks_per_seq, torch.bfloat16)
    assert plan.schedule == 0
    assert_decode_close(to_f64(gpu_decode(inp)), oracle.decode_inputs(inp), "bf16")


TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
