"""GPU parity of the swap copy (pa_swap_blocks) against the oracle: bit-exact.

Swap out (device cache -> pinned host cache), swap in (host -> device, pairs in
pinned host memory), device -> device, every dtype and vector width, bad ids
flagged and skipped, pageable host memory refused; and the preemption round trip
through the block pool: a sequence swapped out and back in decodes to the same
bits as before.
"""
import ctypes
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from helpers import TORCH_DTYPE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    pa.library()
    yield
    pa.check_error()


def _cache(n, h, bs, d, dtype, gen, where):
    bits = torch.randint(-2**15, 2**15, (n, h, bs, d * (2 if dtype == "f32" else 1)), dtype=torch.int16,
                         generator=gen)
    t = bits.view(TORCH_DTYPE[dtype]) if dtype != "f32" else bits.view(torch.float32)
    if where == "host":
        return t.pin_memory()
    return t.cuda()


def _np(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype,h,bs,d", [("bf16", 4, 16, 128), ("f16", 3, 32, 64), ("f32", 2, 16, 64),
                                          ("bf16", 1, 8, 8)])
@pytest.mark.parametrize("direction", ["out", "in", "d2d"])
def test_swap_blocks_bit_exact(dtype, h, bs, d, direction):
    gen = torch.Generator().manual_seed(zlib.crc32(repr((dtype, h, bs, d, direction)).encode()))
    src_where, dst_where = {"out": ("dev", "host"), "in": ("host", "dev"), "d2d": ("dev", "dev")}[direction]
    ns, nd = 37, 23
    sk, sv = _cache(ns, h, bs, d, dtype, gen, src_where), _cache(ns, h, bs, d, dtype, gen, src_where)
    dk, dv = _cache(nd, h, bs, d, dtype, gen, dst_where), _cache(nd, h, bs, d, dtype, gen, dst_where)
    rng = np.random.default_rng(ns)
    pairs = np.stack([rng.choice(ns, 17, replace=False), rng.choice(nd, 17, replace=False)], 1).astype(np.int64)
    exp_k, exp_v = _np(dk), _np(dv)
    assert oracle.swap_blocks(exp_k, exp_v, _np(sk), _np(sv), pairs) == oracle.OK
    src_before = (_np(sk), _np(sv))
    p = torch.from_numpy(pairs)
    p = p.pin_memory() if direction == "in" else p.cuda()
    pa.swap_blocks(dk, dv, sk, sv, p)
    torch.cuda.synchronize()
    assert np.array_equal(_np(dk), exp_k) and np.array_equal(_np(dv), exp_v)
    assert np.array_equal(_np(sk), src_before[0]) and np.array_equal(_np(sv), src_before[1])
    pa.check_error()


def test_swap_blocks_bad_ids_are_skipped_and_flagged():
    gen = torch.Generator().manual_seed(5)
    sk, sv = _cache(4, 2, 16, 64, "bf16", gen, "dev"), _cache(4, 2, 16, 64, "bf16", gen, "dev")
    dk, dv = _cache(3, 2, 16, 64, "bf16", gen, "host"), _cache(3, 2, 16, 64, "bf16", gen, "host")
    pairs = np.array([[0, 1], [4, 0], [1, 3], [-1, 2], [3, 2]], np.int64)
    exp_k, exp_v = _np(dk), _np(dv)
    assert oracle.swap_blocks(exp_k, exp_v, _np(sk), _np(sv), pairs) == oracle.BAD_TABLE
    pa.swap_blocks(dk, dv, sk, sv, torch.from_numpy(pairs).cuda())
    with pytest.raises(pa.PAError) as e:
        pa.check_error()
    assert e.value.status == 5  # PA_ERR_BAD_TABLE
    assert np.array_equal(_np(dk), exp_k) and np.array_equal(_np(dv), exp_v)


def test_swap_blocks_refuses_pageable_host_memory():
    lib = pa.library()
    dk = torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    pageable = np.zeros(2 * 16 * 64, np.uint16)
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    addr = pageable.ctypes.data
    st = lib.pa_swap_blocks(dk.data_ptr(), dk.data_ptr(), addr, addr, pairs.data_ptr(), 1, 1, 64, 16, 2, 2, 2,
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 1 and b"pageable" in lib.pa_last_error_string()
    torch.cuda.synchronize()
    assert int(dk.view(torch.int16).abs().sum()) == 0


def test_preemption_round_trip_decodes_the_same_bits():
    """Fill sequences through the pool, swap one out to a pinned host pool and back in
    (other blocks), and decode: the output bits equal those before the swap."""
    h, hq, bs, d, nb = 2, 8, 16, 128, 64
    torch.manual_seed(0)
    dev_pool, host_pool = pa.BlockPool(nb, bs), pa.BlockPool(32, bs)
    kc = torch.randn(nb, h, bs, d, device="cuda").to(torch.bfloat16)
    vc = torch.randn(nb, h, bs, d, device="cuda").to(torch.bfloat16)
    hk = torch.zeros(32, h, bs, d, dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    seqs = [dev_pool.create() for _ in range(3)]
    lens = [70, 33, 129]
    for sid, n in zip(seqs, lens):
        for _ in range(n):
            dev_pool.append(sid)
    q = torch.randn(3, hq, d, device="cuda").to(torch.bfloat16)

    def run(ids):
        tables, ctx = dev_pool.block_tables(ids, 16)
        return pa.decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda())

    before = run(seqs).clone()
    hid, out_pairs = dev_pool.swap_to(host_pool, seqs[2])
    pa.swap_blocks(hk, hv, kc, vc, torch.from_numpy(out_pairs).cuda())
    torch.cuda.synchronize()
    # the freed device blocks are reused by someone else meanwhile
    filler = dev_pool.create()
    for _ in range(5 * bs):
        dev_pool.append(filler)
    kc.index_fill_(0, torch.from_numpy(np.unique(out_pairs[:, 0])).cuda(), float("nan"))
    back, in_pairs = host_pool.swap_to(dev_pool, hid)
    in_pairs_host = torch.from_numpy(in_pairs).pin_memory()  # kept alive until the stream has read it
    pa.swap_blocks(kc, vc, hk, hv, in_pairs_host)
    after = run([seqs[0], seqs[1], back])
    torch.cuda.synchronize()
    dev_pool.check_invariants()
    host_pool.check_invariants()
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
    pa.check_error()
