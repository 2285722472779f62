"""GPU parity of pa_decode_append (the new token written at position L - 1, then
attended) against the oracle: the cache bit-exact after the oracle's write at the
slots the block tables give position L - 1, the output within the decode
tolerance of the oracle's decode over the written cache, and bit-identical to
pa_write_kv followed by pa_decode with the same plan.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from paged_kv_cache_129_gb300 import workloads as wl
from helpers import TORCH_DTYPE, assert_decode_close, to_device, to_f64, to_host
from test_gpu_kernels import CASES, RAGGED

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    yield
    pa.check_error()


def append_case(dtype, d, bs, hq, hkv, lens, seed):
    return wl.make_decode_inputs(f"append_{dtype}", context_lens=list(lens), num_heads=hq, num_kv_heads=hkv,
                                 head_dim=d, block_size=bs, dtype=dtype, pool_slack=0.5, seed=seed,
                                 with_new_token=True)


def oracle_step(inp):
    """Oracle: write the new rows at the slots of positions L - 1 (none for L == 0), then decode."""
    live = [b for b in range(inp.num_seqs) if inp.context_lens[b] >= 1]
    slots = np.full(inp.num_seqs, -1, dtype=np.int64)
    slots[live] = oracle.slots_for_positions(inp.block_tables, live, [int(inp.context_lens[b]) - 1 for b in live],
                                             inp.block_size)
    kc, vc = inp.key_cache.copy(), inp.value_cache.copy()
    assert oracle.write_kv(inp.new_key, inp.new_value, kc, vc, slots) == 0
    ref = oracle.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.dtype, inp.scale)
    return kc, vc, ref, slots


def workspace_for(inp, partition_pages, kernel):
    if partition_pages < 0:
        return None
    plan = pa.decode_plan(inp.num_seqs, inp.num_heads, inp.num_kv_heads, inp.head_dim, inp.block_size,
                          inp.max_blocks_per_seq, TORCH_DTYPE[inp.dtype], partition_pages=partition_pages,
                          kernel=kernel)
    return torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("dtype,d,bs,hq,hkv,kernel", CASES)
@pytest.mark.parametrize("partition_pages", [0, 3, -1])
def test_append_matches_oracle_and_unfused_path(dtype, d, bs, hq, hkv, kernel, partition_pages):
    seed = zlib.crc32(f"append{dtype}{d}{bs}{hq}{hkv}".encode()) % 1000
    inp = append_case(dtype, d, bs, hq, hkv, RAGGED, seed)
    kc_ref, vc_ref, ref, slots = oracle_step(inp)
    q, nk, nv = to_device(inp.q, dtype), to_device(inp.new_key, dtype), to_device(inp.new_value, dtype)
    bt, lens = torch.from_numpy(inp.block_tables).cuda(), torch.from_numpy(inp.context_lens).cuda()
    ws = workspace_for(inp, partition_pages, kernel)

    kc, vc = to_device(inp.key_cache, dtype), to_device(inp.value_cache, dtype)
    out = pa.decode_append(q, nk, nv, kc, vc, bt, lens, scale=inp.scale, workspace=ws,
                           partition_pages=partition_pages, kernel=kernel)
    torch.cuda.synchronize()
    pa.check_error()
    assert np.array_equal(to_host(kc, dtype), kc_ref) and np.array_equal(to_host(vc, dtype), vc_ref)
    assert_decode_close(to_f64(out), ref, dtype)

    # the unfused path on fresh caches: same bytes in the cache, the same output bits
    kc2, vc2 = to_device(inp.key_cache, dtype), to_device(inp.value_cache, dtype)
    pa.write_kv(nk, nv, kc2, vc2, torch.from_numpy(slots).cuda())
    out2 = pa.decode(q, kc2, vc2, bt, lens, scale=inp.scale, workspace=ws, partition_pages=partition_pages,
                     kernel=kernel)
    torch.cuda.synchronize()
    pa.check_error()
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(out.view(torch.int16) if dtype != "f32" else out,
                       out2.view(torch.int16) if dtype != "f32" else out2)


@pytest.mark.parametrize("partition_pages", [0, -1])
def test_append_qwen_shape_full_and_last_rows(partition_pages):
    # lengths that put the new token on the first, a middle and the last row of a page
    lens = [1, 2, 16, 17, 31, 32, 33, 48, 511, 512, 513, 4096]
    inp = append_case("bf16", 128, 16, 28, 4, lens, seed=5)
    kc_ref, vc_ref, ref, _ = oracle_step(inp)
    kc, vc = to_device(inp.key_cache, "bf16"), to_device(inp.value_cache, "bf16")
    out = pa.decode_append(to_device(inp.q, "bf16"), to_device(inp.new_key, "bf16"), to_device(inp.new_value, "bf16"),
                           kc, vc, torch.from_numpy(inp.block_tables).cuda(), torch.from_numpy(inp.context_lens).cuda(),
                           scale=inp.scale, workspace=workspace_for(inp, partition_pages, "auto"),
                           partition_pages=partition_pages)
    torch.cuda.synchronize()
    pa.check_error()
    assert np.array_equal(to_host(kc, "bf16"), kc_ref) and np.array_equal(to_host(vc, "bf16"), vc_ref)
    assert_decode_close(to_f64(out), ref, "bf16")


def test_append_twice_in_a_row_extends_the_context():
    # step 1 appends at L - 1; step 2, with L + 1, appends the next token and attends to both
    lens = np.array([15, 16, 40, 100], dtype=np.int32)
    inp = append_case("bf16", 128, 16, 8, 2, lens + 1, seed=9)  # tables sized for L + 1
    first = wl.make_decode_inputs("append_first", context_lens=list(lens + 1), num_heads=8, num_kv_heads=2,
                                  head_dim=128, block_size=16, dtype="bf16", pool_slack=0.5, seed=10,
                                  with_new_token=True)
    kc, vc = to_device(inp.key_cache, "bf16"), to_device(inp.value_cache, "bf16")
    bt = torch.from_numpy(inp.block_tables).cuda()
    q = to_device(inp.q, "bf16")
    ws = workspace_for(inp, 0, "auto")
    pa.decode_append(q, to_device(first.new_key, "bf16"), to_device(first.new_value, "bf16"), kc, vc, bt,
                     torch.from_numpy(lens).cuda(), scale=inp.scale, workspace=ws)
    out = pa.decode_append(q, to_device(inp.new_key, "bf16"), to_device(inp.new_value, "bf16"), kc, vc, bt,
                           torch.from_numpy(lens + 1).cuda(), scale=inp.scale, workspace=ws)
    torch.cuda.synchronize()
    pa.check_error()
    # oracle: the two writes, then the decode over L + 1 tokens
    ekc, evc = inp.key_cache.copy(), inp.value_cache.copy()
    seqs = list(range(len(lens)))
    s1 = oracle.slots_for_positions(inp.block_tables, seqs, [int(x) - 1 for x in lens], 16)
    s2 = oracle.slots_for_positions(inp.block_tables, seqs, [int(x) for x in lens], 16)
    assert oracle.write_kv(first.new_key, first.new_value, ekc, evc, s1) == 0
    assert oracle.write_kv(inp.new_key, inp.new_value, ekc, evc, s2) == 0
    assert np.array_equal(to_host(kc, "bf16"), ekc) and np.array_equal(to_host(vc, "bf16"), evc)
    ref = oracle.decode(inp.q, ekc, evc, inp.block_tables, lens + 1, "bf16", inp.scale)
    assert_decode_close(to_f64(out), ref, "bf16")


def test_append_bad_last_block_is_reported_and_not_written():
    inp = append_case("bf16", 128, 16, 8, 2, [20, 33], seed=11)
    tables = inp.block_tables.copy()
    tables[1, 2] = inp.num_blocks + 7  # the page holding position 32 of sequence 1
    kc, vc = to_device(inp.key_cache, "bf16"), to_device(inp.value_cache, "bf16")
    pa.decode_append(to_device(inp.q, "bf16"), to_device(inp.new_key, "bf16"), to_device(inp.new_value, "bf16"),
                     kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(inp.context_lens).cuda(),
                     scale=inp.scale, workspace=workspace_for(inp, 0, "auto"))
    with pytest.raises(pa.PAError) as err:
        pa.check_error()
    assert err.value.status == 5  # PA_ERR_BAD_TABLE
    # sequence 0's row is written; nothing else in the caches changed
    ekc, evc = inp.key_cache.copy(), inp.value_cache.copy()
    s0 = oracle.slots_for_positions(tables, [0], [19], 16)
    assert oracle.write_kv(inp.new_key[:1], inp.new_value[:1], ekc, evc, s0) == 0
    assert np.array_equal(to_host(kc, "bf16"), ekc) and np.array_equal(to_host(vc, "bf16"), evc)


def test_append_rejects_misaligned_new_rows():
    inp = append_case("bf16", 128, 16, 8, 2, [5], seed=12)
    flat = torch.zeros(2 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    nk = flat[1:1 + 2 * 128].view(1, 2, 128)  # 2-byte offset
    with pytest.raises(pa.PAError):
        pa.decode_append(to_device(inp.q, "bf16"), nk, nk, to_device(inp.key_cache, "bf16"),
                         to_device(inp.value_cache, "bf16"), torch.from_numpy(inp.block_tables).cuda(),
                         torch.from_numpy(inp.context_lens).cuda())
