"""Pins for the multi-query (verify) oracle: sequence b's q_len query tokens sit at positions
L - q_len .. L - 1 and token t attends positions 0 .. L - q_len + t.

* textbook routine: causal softmax attention (scipy) on K/V gathered contiguously by numpy;
* reductions: q_len = 1 is the single-query decode; the last token is the single-query decode over
  the whole context; token 0 of a context of exactly q_len tokens returns v_0;
* invariants: a permutation of the physical blocks; K/V past a token's causal bound (poisoned with
  huge values) does not reach it; bounds below 0 give zero rows.
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from paged_kv_cache_129_gb300 import workloads as wl


def to_f64(arr, dtype):
    if dtype in ("f32", "f16"):
        return arr.astype(np.float64)
    return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def case(dtype="bf16", lens=(3, 7, 16, 17, 40, 64), q_len=3, hq=6, hkv=2, d=32, bs=16, seed=0, slack=0.5):
    return wl.make_decode_inputs(f"mq_{dtype}", context_lens=list(lens), num_heads=hq, num_kv_heads=hkv, head_dim=d,
                                 block_size=bs, dtype=dtype, pool_slack=slack, seed=seed, q_len=q_len)


def run(inp):
    return oracle.decode_multi(inp.q, inp.key_cache, inp.value_cache, inp.block_tables, inp.context_lens, inp.dtype,
                               inp.scale)


def dense_causal(inp):
    kc, vc, q = (to_f64(x, inp.dtype) for x in (inp.key_cache, inp.value_cache, inp.q))
    B, n, Hq, d = q.shape
    g = Hq // inp.num_kv_heads
    out = np.zeros_like(q)
    for b in range(B):
        L = int(inp.context_lens[b])
        if L == 0:
            continue
        pages = inp.block_tables[b, :-(-L // inp.block_size)]
        for kvh in range(inp.num_kv_heads):
            K = kc[pages, kvh].reshape(-1, d)[:L]
            V = vc[pages, kvh].reshape(-1, d)[:L]
            for t in range(n):
                pos = L - n + t  # the token's own position
                if pos < 0:
                    continue
                S = q[b, t, kvh * g:(kvh + 1) * g] @ K.T * inp.scale  # [g, L]
                S[:, pos + 1:] = -np.inf                               # causal mask
                out[b, t, kvh * g:(kvh + 1) * g] = softmax(S, axis=-1) @ V
    return out


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("q_len,bs", [(2, 16), (3, 4), (5, 16), (8, 1)])
def test_matches_dense_causal_attention(dtype, q_len, bs):
    inp = case(dtype, q_len=q_len, bs=bs, seed=q_len * 10 + bs)
    np.testing.assert_allclose(run(inp), dense_causal(inp), rtol=1e-12, atol=1e-12)


def test_q_len_one_is_the_decode():
    inp = case(q_len=2, seed=4)
    one = wl.make_decode_inputs("one", context_lens=list(inp.context_lens), num_heads=6, num_kv_heads=2, head_dim=32,
                                block_size=16, dtype="bf16", pool_slack=0.5, seed=4)
    got = oracle.decode_multi(one.q[:, None], one.key_cache, one.value_cache, one.block_tables, one.context_lens,
                              "bf16", one.scale)
    np.testing.assert_array_equal(got[:, 0], oracle.decode_inputs(one))


def test_last_token_is_the_single_decode_over_the_context():
    inp = case(q_len=4, seed=6)
    got = run(inp)
    single = oracle.decode(np.ascontiguousarray(inp.q[:, -1]), inp.key_cache, inp.value_cache, inp.block_tables,
                           inp.context_lens, "bf16", inp.scale)
    np.testing.assert_allclose(got[:, -1], single, rtol=1e-13, atol=1e-13)


def test_first_token_of_a_context_of_q_len_tokens_returns_v0():
    inp = case("f32", lens=(4, 4), q_len=4, seed=8)
    got = run(inp)
    vc = inp.value_cache
    g = 3
    for b in range(2):
        pb = int(inp.block_tables[b, 0])
        for qh in range(6):
            np.testing.assert_array_equal(got[b, 0, qh], vc[pb, qh // g, 0].astype(np.float64))


def test_rows_before_the_context_start_are_zero():
    inp = case(lens=(1, 2, 0, 9), q_len=3, seed=9)
    got = run(inp)
    assert not got[0, :2].any() and got[0, 2].any()   # L=1: only the last token has a position
    assert not got[1, 0].any() and got[1, 1:].any()   # L=2
    assert not got[2].any()                           # L=0


def test_invariant_under_physical_block_permutation():
    inp = case(q_len=3, seed=13, slack=1.0)
    base = run(inp)
    pi = np.random.default_rng(1).permutation(inp.num_blocks)
    kc, vc = np.empty_like(inp.key_cache), np.empty_like(inp.value_cache)
    kc[pi], vc[pi] = inp.key_cache, inp.value_cache
    tables = np.where(inp.block_tables >= 0, pi[np.maximum(inp.block_tables, 0)], -1).astype(np.int32)
    got = oracle.decode_multi(inp.q, kc, vc, tables, inp.context_lens, "bf16", inp.scale)
    np.testing.assert_allclose(got, base, rtol=1e-13, atol=1e-13)


def test_positions_past_a_tokens_bound_do_not_reach_it():
    inp = case("f32", lens=(20, 33), q_len=4, seed=14)
    base = run(inp)
    kc, vc = inp.key_cache.copy(), inp.value_cache.copy()
    # poison the last position of every sequence: only token q_len - 1 may see it
    for b, L in enumerate(inp.context_lens):
        pos = int(L) - 1
        pb = int(inp.block_tables[b, pos // inp.block_size])
        kc[pb, :, pos % inp.block_size] = 1e3
        vc[pb, :, pos % inp.block_size] = 1e6
    got = oracle.decode_multi(inp.q, kc, vc, inp.block_tables, inp.context_lens, "f32", inp.scale)
    np.testing.assert_array_equal(got[:, :-1], base[:, :-1])
    assert np.abs(got[:, -1] - base[:, -1]).max() > 1.0
