"""GPU parity on the five workloads at full size, in the launch configuration
the benchmark times (default plan, workspace sized by pa_decode_workspace_size).

qwen_gqa, mha_short (bs 16 and 32) and prefix_cow: every output row against
the oracle.  long_context: 48 sampled rows (all heads of the longest sequence
plus 16 random rows), since the oracle walks ~0.5 M tokens per head.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from oracle.block_pool import SequencePool
from paged_kv_cache_129_gb300 import workloads as wl
from helpers import TORCH_DTYPE, assert_decode_close, slots_of, to_device, to_f64, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    yield
    pa.check_error()


def run_default(inp, dev):
    ws_bytes = pa.decode_workspace_size(inp.num_seqs, inp.num_heads, inp.num_kv_heads, inp.head_dim,
                                        inp.block_size, inp.max_blocks_per_seq, TORCH_DTYPE[inp.dtype])
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = pa.decode(dev["q"], dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws)
    torch.cuda.synchronize()
    pa.check_error()
    return out


def upload(inp):
    return dict(q=to_device(inp.q, inp.dtype), kc=to_device(inp.key_cache, inp.dtype),
                vc=to_device(inp.value_cache, inp.dtype), bt=torch.from_numpy(inp.block_tables).cuda(),
                lens=torch.from_numpy(inp.context_lens).cuda())


def test_qwen_gqa_write_then_decode():
    inp = wl.qwen_gqa()
    dev = upload(inp)
    slots = slots_of(inp.block_tables, range(inp.num_seqs), inp.new_token_pos, inp.block_size)
    pa.write_kv(to_device(inp.new_key, "bf16"), to_device(inp.new_value, "bf16"), dev["kc"], dev["vc"],
                torch.from_numpy(slots).cuda())
    got = to_f64(run_default(inp, dev))
    # the written rows are bit-exact
    assert oracle.write_kv(inp.new_key, inp.new_value, inp.key_cache, inp.value_cache, slots) == 0
    blocks = np.unique(slots // inp.block_size)
    assert np.array_equal(to_host(dev["kc"][torch.from_numpy(blocks).cuda()], "bf16"), inp.key_cache[blocks])
    assert np.array_equal(to_host(dev["vc"][torch.from_numpy(blocks).cuda()], "bf16"), inp.value_cache[blocks])
    assert_decode_close(got, oracle.decode_inputs(inp), "bf16")


def test_long_context_sampled_rows():
    inp = wl.long_context()
    got = to_f64(run_default(inp, upload(inp)))
    longest = int(np.argmax(inp.context_lens))
    rng = np.random.default_rng(1)
    rows = [(longest, h) for h in range(inp.num_heads)]
    rows += [(int(b), int(h)) for b, h in zip(rng.integers(0, inp.num_seqs, 16), rng.integers(0, inp.num_heads, 16))]
    ref = oracle.decode_inputs(inp, rows=rows)
    assert_decode_close(np.stack([got[b, h] for b, h in rows]), ref, "bf16")


@pytest.mark.parametrize("block_size", [16, 32])
def test_mha_short(block_size):
    inp = wl.mha_short(block_size)
    got = to_f64(run_default(inp, upload(inp)))
    assert_decode_close(got, oracle.decode_inputs(inp), "f16")


@pytest.mark.parametrize("prefix_len,expected_copies", [(2048, 0), (2056, 63)])
def test_prefix_sharing_with_copy_on_write(prefix_len, expected_copies):
    w = wl.prefix_cow(prefix_len=prefix_len)
    bs = w.block_size
    # product pool (GPU side) and allocator model (oracle side), driven identically
    pool = pa.BlockPool(w.num_blocks, bs)
    model = SequencePool(w.num_blocks, bs)
    parent, mparent = pool.create(), model.create()
    for _ in range(prefix_len):
        pool.append(parent)
        model.append(mparent)
    seqs = [parent] + [pool.fork(parent) for _ in range(w.num_seqs - 1)]
    mseqs = [mparent] + [model.fork(mparent) for _ in range(w.num_seqs - 1)]
    slots, pairs, mslots, mpairs = [], [], [], []
    for sid, mid, tail in zip(seqs, mseqs, w.tail_lens):
        for _ in range(int(tail)):
            s, cow = pool.append(sid)
            r = model.append(mid)
            slots.append(s)
            mslots.append(r.slot)
            if cow:
                pairs.append(cow)
            if r.cow:
                mpairs.append(r.cow)
    assert slots == mslots and pairs == mpairs and len(pairs) == expected_copies
    width = max(len(model.tables[m]) for m in mseqs)
    tables, lens = pool.block_tables(seqs, width)
    mtables, mlens = model.block_tables(mseqs, width)
    assert np.array_equal(tables, mtables) and np.array_equal(lens, mlens)
    pool.check_invariants()

    # GPU: copy the shared tails, write the private tails, decode
    kc, vc = to_device(w.key_cache, "bf16"), to_device(w.value_cache, "bf16")
    if pairs:
        pa.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int64, device="cuda"))
    pa.write_kv(to_device(w.tail_key, "bf16"), to_device(w.tail_value, "bf16"), kc, vc,
                torch.tensor(slots, dtype=torch.int64, device="cuda"))
    q = to_device(w.q, "bf16")
    bt, dl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    ws_bytes = pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, bs, width,
                                        torch.bfloat16)
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = pa.decode(q, kc, vc, bt, dl, scale=wl.default_scale(w.head_dim), workspace=ws)
    torch.cuda.synchronize()
    pa.check_error()

    # oracle: same steps on host copies, with the model's own pairs and slots
    ekc, evc = w.key_cache.copy(), w.value_cache.copy()
    if mpairs:
        assert oracle.copy_blocks(ekc, evc, np.array(mpairs)) == 0
    assert oracle.write_kv(w.tail_key, w.tail_value, ekc, evc, np.array(mslots, dtype=np.int64)) == 0
    assert np.array_equal(to_host(kc, "bf16"), ekc) and np.array_equal(to_host(vc, "bf16"), evc)
    ref = oracle.decode(w.q, ekc, evc, mtables, mlens, "bf16", wl.default_scale(w.head_dim))
    assert_decode_close(to_f64(out), ref, "bf16")
