"""GPU: pa.DecodeStepper (packed pinned uploads, two slots in flight) gives the same bytes as the
direct calls, step by step, with steps overlapping on the GPU."""
import numpy as np
import pytest
import torch

import paged_kv_cache_129_gb300 as pa
from paged_kv_cache_129_gb300 import workloads as wl
from helpers import TORCH_DTYPE, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    yield
    pa.check_error()


def host(arr, dtype):
    a = np.ascontiguousarray(arr)
    t = torch.from_numpy(a.view(np.int16) if dtype in ("bf16", "f16") else a)
    return t.view(TORCH_DTYPE[dtype]) if dtype in ("bf16", "f16") else t


@pytest.mark.parametrize("append", [True, False])
@pytest.mark.parametrize("dtype,hq,hkv,lens", [
    ("bf16", 28, 4, [1, 17, 300, 1000, 2049, 33]),   # lean schedule
    ("f16", 32, 32, [16, 40, 100, 200] * 32),          # partitioned grid, one pass
])
def test_stepper_matches_direct_calls(append, dtype, hq, hkv, lens):
    steps = 5
    batches = [wl.make_decode_inputs("step", context_lens=lens, num_heads=hq, num_kv_heads=hkv, head_dim=128,
                                     block_size=16, dtype=dtype, pool_slack=0.5, seed=s, with_new_token=True)
               for s in range(steps)]
    base = batches[0]  # caches and tables of step 0 serve every step; q and new K/V differ per step
    kc, vc = to_device(base.key_cache, dtype), to_device(base.value_cache, dtype)
    kc_ref, vc_ref = kc.clone(), vc.clone()
    bt = torch.from_numpy(base.block_tables)
    ln = torch.from_numpy(base.context_lens)
    stepper = pa.DecodeStepper(kc, vc, base.num_seqs, hq, base.max_blocks_per_seq, scale=base.scale,
                               append=append)
    got = []
    for i in range(steps):
        if i >= stepper.slots:
            got.append(stepper.result(i - stepper.slots).clone())
        v = stepper.inputs(i)
        v.query.copy_(host(batches[i].q, dtype))
        v.block_tables.copy_(bt)
        v.context_lens.copy_(ln)
        if append:
            v.new_key.copy_(host(batches[i].new_key, dtype))
            v.new_value.copy_(host(batches[i].new_value, dtype))
        stepper.launch(i)
    for i in range(steps - stepper.slots, steps):
        got.append(stepper.result(i).clone())
    torch.cuda.synchronize()
    pa.check_error()

    ws_bytes = pa.decode_workspace_size(base.num_seqs, hq, hkv, 128, 16, base.max_blocks_per_seq,
                                        TORCH_DTYPE[dtype])
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda") if ws_bytes else None
    btd, lnd = bt.cuda(), ln.cuda()
    for i in range(steps):
        q = to_device(batches[i].q, dtype)
        if append:
            ref = pa.decode_append(q, to_device(batches[i].new_key, dtype), to_device(batches[i].new_value, dtype),
                                   kc_ref, vc_ref, btd, lnd, scale=base.scale, workspace=ws)
        else:
            ref = pa.decode(q, kc_ref, vc_ref, btd, lnd, scale=base.scale, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got[i].view(torch.int16), ref.cpu().view(torch.int16)), f"step {i}"
    assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref)
    pa.check_error()


def test_stepper_with_table_deltas_matches_full_tables():
    """Sequences grow by one token a step through the block pool (new blocks, a fork's
    copy-on-write tail); the stepper keeps the device tables current with the pool's delta
    exports only, and every step's output and the caches equal direct pa_decode_append calls
    given the full tables."""
    rng = np.random.default_rng(5)
    nb, hkv, hq, bs, d, B, width, steps = 300, 4, 28, 16, 128, 6, 24, 40
    pool = pa.BlockPool(nb, bs, free_order=rng.permutation(nb))
    seqs = [pool.create() for _ in range(B - 1)]
    for sid, n in zip(seqs, rng.integers(1, 200, B - 1)):
        for _ in range(int(n)):
            pool.append(sid)
    seqs.append(pool.fork(seqs[0]))  # shares seqs[0]'s blocks; its first append copies a partial tail
    kc = torch.randn(nb, hkv, bs, d, device="cuda").to(torch.bfloat16)
    vc = torch.randn(nb, hkv, bs, d, device="cuda").to(torch.bfloat16)
    kc_ref, vc_ref = kc.clone(), vc.clone()
    stepper = pa.DecodeStepper(kc, vc, B, hq, width, append=True, tables="deltas")
    # the same plan as the stepper's (its workspace size), so the direct calls take the same schedule
    ws_bytes = pa.decode_workspace_size(B, hq, hkv, d, bs, width, torch.bfloat16)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda") if ws_bytes else None
    got, refs, sent = [], [], []
    for i in range(steps):
        if i >= stepper.slots:
            got.append(stepper.result(i - stepper.slots).clone())
        cow = []
        for sid in seqs:
            _, pair = pool.append(sid)
            if pair:
                cow.append(pair)
        if cow:  # the copy-on-write copies, on both caches, before this step's decode
            pairs = torch.tensor(cow, dtype=torch.int64, device="cuda")
            pa.copy_blocks(kc, vc, pairs)
            pa.copy_blocks(kc_ref, vc_ref, pairs)
        v = stepper.inputs(i)
        deltas, lens = pool.table_deltas(seqs, out=v.deltas.numpy(), lens_out=v.context_lens.numpy())
        sent.append(len(deltas))
        if i == 0:
            entries0 = sum((pool.length(sid) + bs - 1) // bs for sid in seqs)
        q = torch.randn(B, hq, d).to(torch.bfloat16)
        nk = torch.randn(B, hkv, d).to(torch.bfloat16)
        nv = torch.randn(B, hkv, d).to(torch.bfloat16)
        v.query.copy_(q)
        v.new_key.copy_(nk)
        v.new_value.copy_(nv)
        stepper.launch(i, num_deltas=len(deltas))
        full, full_lens = pool.block_tables(seqs, width)
        refs.append(pa.decode_append(q.cuda(), nk.cuda(), nv.cuda(), kc_ref, vc_ref, torch.from_numpy(full).cuda(),
                                     torch.from_numpy(full_lens).cuda(), workspace=ws))
    for i in range(steps - stepper.slots, steps):
        got.append(stepper.result(i).clone())
    torch.cuda.synchronize()
    pa.check_error()
    for i in range(steps):
        assert torch.equal(got[i].view(torch.int16), refs[i].cpu().view(torch.int16)), f"step {i}"
    assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref)
    # the first step sends every entry; later steps only the new blocks and copied tails
    assert sent[0] == entries0
    assert max(sent[1:]) <= B and sum(sent[1:]) < steps * B / 4
