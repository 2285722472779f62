"""Pins for the fp64 decode oracle, each against something other than the oracle itself.

* textbook routine: dense softmax attention (scipy) on K/V gathered contiguously
  through numpy fancy indexing, with elements decoded by numpy/torch casts;
* invariants: a permutation of the physical blocks; NaN garbage in masked tail
  slots and unused blocks; the GQA head mapping (unmapped kv heads poisoned);
* hand-worked cases: L = 1, identical keys, q = 0, a dominant key, and the
  two-token fixture under tests/golden;
* the per-block-softmax variant printed on the PagedAttention source-analysis
  page must differ from the method whenever a context spans several blocks.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from paged_kv_cache_129_gb300 import workloads as wl


def to_f64(arr, dtype):
    """Library decoding of the storage forms (independent of the oracle's C decoder)."""
    if dtype == "f32":
        return arr.astype(np.float64)
    if dtype == "f16":
        return arr.astype(np.float64)
    return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def dense_reference(inp):
    """softmax(q K^T * scale) V per (b, qh), on K/V gathered into contiguous arrays."""
    kc = to_f64(inp.key_cache, inp.dtype)
    vc = to_f64(inp.value_cache, inp.dtype)
    q = to_f64(inp.q, inp.dtype)
    B, Hq, d = q.shape
    g = Hq // inp.num_kv_heads
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = int(inp.context_lens[b])
        if L == 0:
            continue
        nblk = -(-L // inp.block_size)
        pages = inp.block_tables[b, :nblk]
        for kvh in range(inp.num_kv_heads):
            K = kc[pages, kvh].reshape(-1, d)[:L]  # [L, d], contiguous copy of the pages
            V = vc[pages, kvh].reshape(-1, d)[:L]
            Q = q[b, kvh * g:(kvh + 1) * g]  # [g, d]
            P = softmax(Q @ K.T * inp.scale, axis=-1)
            out[b, kvh * g:(kvh + 1) * g] = P @ V
    return out


def small_case(dtype, seed, lens=(1, 7, 16, 17, 40, 64), hq=6, hkv=2, d=32, bs=16, slack=0.5):
    return wl.make_decode_inputs(f"small_{dtype}", context_lens=list(lens), num_heads=hq, num_kv_heads=hkv,
                                 head_dim=d, block_size=bs, dtype=dtype, pool_slack=slack, seed=seed)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("bs", [1, 4, 16])
def test_matches_dense_softmax_attention(dtype, bs):
    inp = small_case(dtype, seed=11 + bs, bs=bs)
    ref = dense_reference(inp)
    got = oracle.decode_inputs(inp)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_tiny_workload_matches_dense():
    inp = wl.tiny()
    np.testing.assert_allclose(oracle.decode_inputs(inp), dense_reference(inp), rtol=1e-12, atol=1e-12)


def test_invariant_under_physical_block_permutation():
    inp = small_case("bf16", seed=3, slack=1.0)
    base = oracle.decode_inputs(inp)
    pi = np.random.default_rng(5).permutation(inp.num_blocks)
    kc = np.empty_like(inp.key_cache)
    vc = np.empty_like(inp.value_cache)
    kc[pi] = inp.key_cache  # block i moves to pi[i]
    vc[pi] = inp.value_cache
    bt = np.where(inp.block_tables >= 0, pi[np.maximum(inp.block_tables, 0)], -1).astype(np.int32)
    moved = oracle.decode(inp.q, kc, vc, bt, inp.context_lens, inp.dtype, inp.scale)
    np.testing.assert_allclose(moved, base, rtol=1e-14, atol=1e-14)


def test_masked_tail_and_unused_blocks_do_not_matter():
    inp = small_case("f32", seed=4, lens=(3, 15, 17, 31), slack=1.0)
    base = oracle.decode_inputs(inp)
    kc, vc = inp.key_cache.copy(), inp.value_cache.copy()
    used = set()
    for b, L in enumerate(inp.context_lens):
        nblk = -(-int(L) // inp.block_size)
        used.update(int(x) for x in inp.block_tables[b, :nblk])
        last = inp.block_tables[b, nblk - 1]
        tail = int(L) - (nblk - 1) * inp.block_size
        kc[last, :, tail:, :] = np.nan
        vc[last, :, tail:, :] = np.inf
    for blk in range(inp.num_blocks):
        if blk not in used:
            kc[blk] = np.nan
            vc[blk] = np.nan
    got = oracle.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, "f32", inp.scale)
    assert np.isfinite(got).all()
    np.testing.assert_array_equal(got, base)


def test_gqa_mapping_uses_floor_division():
    # 8 q heads on 2 kv heads: q heads 0-3 read kv head 0 only. Poison kv head 1.
    inp = small_case("f32", seed=6, lens=(5, 20), hq=8, hkv=2)
    kc, vc = inp.key_cache.copy(), inp.value_cache.copy()
    kc[:, 1] = np.nan
    vc[:, 1] = np.nan
    got = oracle.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, "f32", inp.scale)
    assert np.isfinite(got[:, :4]).all()
    assert np.isnan(got[:, 4:]).all()
    np.testing.assert_allclose(got[:, :4], dense_reference(inp)[:, :4], rtol=1e-12, atol=1e-12)


def test_context_length_one_returns_first_value_exactly():
    inp = small_case("f16", seed=7, lens=(1, 1, 1))
    got = oracle.decode_inputs(inp)
    g = inp.num_heads // inp.num_kv_heads
    for b in range(3):
        pb = inp.block_tables[b, 0]
        for qh in range(inp.num_heads):
            v0 = inp.value_cache[pb, qh // g, 0].astype(np.float64)
            np.testing.assert_array_equal(got[b, qh], v0)


def test_identical_keys_and_zero_query_give_mean_value():
    inp = small_case("f32", seed=8, lens=(9, 33))
    # identical keys: every key row of every block is the same vector
    kc = np.broadcast_to(inp.key_cache[0, 0, 0], inp.key_cache.shape).copy()
    got = oracle.decode(inp.q, kc, inp.value_cache, inp.block_tables, inp.context_lens, "f32", inp.scale)
    zero_q = oracle.decode(np.zeros_like(inp.q), inp.key_cache, inp.value_cache, inp.block_tables,
                           inp.context_lens, "f32", inp.scale)
    g = inp.num_heads // inp.num_kv_heads
    for b, L in enumerate(inp.context_lens):
        nblk = -(-int(L) // inp.block_size)
        for qh in range(inp.num_heads):
            V = inp.value_cache[inp.block_tables[b, :nblk], qh // g].reshape(-1, inp.head_dim)[:L]
            mean = V.astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(got[b, qh], mean, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(zero_q[b, qh], mean, rtol=1e-13, atol=1e-13)


def test_dominant_key_selects_its_value():
    d, L, bs = 8, 37, 16
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 1.0
    nb = 3
    kc = np.zeros((nb, 1, bs, d), np.float32)
    vc = np.random.default_rng(9).standard_normal((nb, 1, bs, d)).astype(np.float32)
    bt = np.array([[2, 0, 1]], np.int32)
    # logical position 20 -> block 0 (table slot 1), offset 4
    kc[0, 0, 4, 0] = 100.0
    got = oracle.decode(q, kc, vc, bt, np.array([L], np.int32), "f32", 1.0)
    np.testing.assert_allclose(got[0, 0], vc[0, 0, 4], rtol=0, atol=1e-40 + 40 * math.exp(-100.0))


def test_large_scores_stay_finite():
    # scores of several thousand overflow exp() in double unless the maximum is subtracted first
    inp = small_case("f32", seed=10, lens=(16, 40))
    q = (inp.q * 2000).astype(np.float32)
    got = oracle.decode(q, inp.key_cache, inp.value_cache, inp.block_tables, inp.context_lens, "f32", inp.scale)
    assert np.isfinite(got).all()
    inp.q = q
    np.testing.assert_allclose(got, dense_reference(inp), rtol=1e-10, atol=1e-10)


def test_zero_context_gives_zero_row():
    inp = small_case("bf16", seed=12, lens=(0, 5, 0))
    got = oracle.decode_inputs(inp)
    assert (got[0] == 0).all() and (got[2] == 0).all()
    assert np.abs(got[1]).sum() > 0


def test_two_token_golden(golden_dir):
    with open(os.path.join(golden_dir, "two_token_decode.json")) as f:
        fx = json.load(f)
    nb, bs, d = fx["num_blocks"], fx["block_size"], fx["head_dim"]
    kc = np.full((nb, 1, bs, d), np.nan, np.float32)
    vc = np.full((nb, 1, bs, d), np.nan, np.float32)
    for blk, row in fx["key_blocks"].items():
        kc[int(blk), 0, 0] = row
    for blk, row in fx["value_blocks"].items():
        vc[int(blk), 0, 0] = row
    q = np.array(fx["q"], np.float32)
    got = oracle.decode(q, kc, vc, np.array(fx["block_table"], np.int32), np.array(fx["context_lens"], np.int32),
                        "f32", math.log(3.0))
    np.testing.assert_allclose(got, np.array(fx["expected"]), rtol=0, atol=1e-14)


def per_block_softmax(inp):
    """The per-block softmax then sum of block outputs (the source-analysis page's loop)."""
    kc, vc, q = (to_f64(x, inp.dtype) for x in (inp.key_cache, inp.value_cache, inp.q))
    B, Hq, d = q.shape
    g = Hq // inp.num_kv_heads
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = int(inp.context_lens[b])
        for lb in range(-(-L // inp.block_size)):
            pb = inp.block_tables[b, lb]
            valid = min(inp.block_size, L - lb * inp.block_size)
            for qh in range(Hq):
                K = kc[pb, qh // g, :valid]
                V = vc[pb, qh // g, :valid]
                out[b, qh] += softmax(K @ q[b, qh] * inp.scale) @ V
    return out


def test_differs_from_per_block_softmax():
    inp = small_case("f32", seed=13, lens=(16, 40, 64))
    got = oracle.decode_inputs(inp)
    wrong = per_block_softmax(inp)
    # one block: identical; several blocks: far apart
    np.testing.assert_allclose(got[0], wrong[0], rtol=1e-12, atol=1e-12)
    assert np.abs(got[1:] - wrong[1:]).max() > 0.5


def test_bad_table_entry_is_reported():
    inp = small_case("f32", seed=14, lens=(20,))
    bt = inp.block_tables.copy()
    bt[0, 1] = inp.num_blocks  # out of the pool
    with pytest.raises(ValueError):
        oracle.decode(inp.q, inp.key_cache, inp.value_cache, bt, inp.context_lens, "f32", inp.scale)


def test_element_decoding_matches_library_casts():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = oracle.element_to_double(bits, "f16")
    lib16 = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(lib16)
    assert (np.isnan(f16) == nan).all()
    np.testing.assert_array_equal(f16[~nan], lib16[~nan])
    bf = oracle.element_to_double(bits, "bf16")
    libbf = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(libbf)
    assert (np.isnan(bf) == nan).all()
    np.testing.assert_array_equal(bf[~nan], libbf[~nan])


def test_row_selection_matches_full_output():
    inp = small_case("bf16", seed=15)
    full = oracle.decode_inputs(inp)
    rows = [(0, 5), (3, 1), (5, 0), (2, 4)]
    part = oracle.decode_inputs(inp, rows=rows)
    for i, (b, h) in enumerate(rows):
        np.testing.assert_array_equal(part[i], full[b, h])
