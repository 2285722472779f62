"""GPU parity of pa_decode_multi (q_len query tokens per sequence, causal) against the oracle.

Query token t of sequence b sits at position L_b - q_len + t and attends positions up to its own;
a token whose position is negative gets a zero row.  Tolerances as for the decode: fp32 1e-5,
bf16/fp16 2e-2 + 1e-2 |ref|.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from paged_kv_cache_129_gb300 import workloads as wl
from helpers import TORCH_DTYPE, assert_decode_close, to_device, to_f64
from test_gpu_kernels import CASES

pytestmark = pytest.mark.gpu

LENS = (0, 1, 2, 3, 15, 16, 17, 33, 100, 257, 700)


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    yield
    pa.check_error()


def mq_case(dtype, d, bs, hq, hkv, q_len, lens=LENS, seed=0):
    return wl.make_decode_inputs(f"mq_{dtype}", context_lens=list(lens), num_heads=hq, num_kv_heads=hkv, head_dim=d,
                                 block_size=bs, dtype=dtype, pool_slack=0.5, seed=seed, q_len=q_len)


def run_multi(inp, partition_pages=0, kernel="auto"):
    q_len = inp.q.shape[1]
    ws = None
    if partition_pages >= 0:
        n = pa.decode_multi_workspace_size(inp.num_seqs, q_len, inp.num_heads, inp.num_kv_heads, inp.head_dim,
                                           inp.block_size, inp.max_blocks_per_seq, TORCH_DTYPE[inp.dtype])
        # partitions of a fixed size may need more than the default plan: give them plenty
        ws = torch.empty(max(n, 64 << 20), dtype=torch.uint8, device="cuda")
    out = pa.decode_multi(to_device(inp.q, inp.dtype), to_device(inp.key_cache, inp.dtype),
                          to_device(inp.value_cache, inp.dtype), torch.from_numpy(inp.block_tables).cuda(),
                          torch.from_numpy(inp.context_lens).cuda(), scale=inp.scale, workspace=ws,
                          partition_pages=partition_pages, kernel=kernel)
    torch.cuda.synchronize()
    pa.check_error()
    return to_f64(out)


def oracle_multi(inp):
    return oracle.decode_multi(inp.q, inp.key_cache, inp.value_cache, inp.block_tables, inp.context_lens, inp.dtype,
                               inp.scale)


@pytest.mark.parametrize("dtype,d,bs,hq,hkv,kernel", CASES)
@pytest.mark.parametrize("q_len", [2, 4])
@pytest.mark.parametrize("partition_pages", [0, 3, -1])
def test_multi_matches_oracle(dtype, d, bs, hq, hkv, kernel, q_len, partition_pages):
    seed = zlib.crc32(f"mq{dtype}{d}{bs}{hq}{hkv}{q_len}".encode()) % 1000
    inp = mq_case(dtype, d, bs, hq, hkv, q_len, seed=seed)
    assert_decode_close(run_multi(inp, partition_pages, kernel).reshape(-1, d),
                        oracle_multi(inp).reshape(-1, d), dtype)


@pytest.mark.parametrize("q_len", [3, 7, 9, 16])
def test_multi_many_rows_per_kv_head(q_len):
    # g * q_len rows per kv head: up to 16 * 7 = 112 rows, i.e. many row chunks per kv head
    inp = mq_case("bf16", 128, 16, 28, 4, q_len, lens=(q_len - 1, q_len, 40, 513, 2000), seed=q_len)
    assert_decode_close(run_multi(inp).reshape(-1, 128), oracle_multi(inp).reshape(-1, 128), "bf16")


def test_q_len_one_is_pa_decode_bit_for_bit():
    inp = mq_case("bf16", 128, 16, 28, 4, 1, seed=3)
    inp.q = np.ascontiguousarray(inp.q)
    q1 = wl.make_decode_inputs("one", context_lens=list(LENS), num_heads=28, num_kv_heads=4, head_dim=128,
                               block_size=16, dtype="bf16", pool_slack=0.5, seed=3)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    dev = dict(kc=to_device(q1.key_cache, "bf16"), vc=to_device(q1.value_cache, "bf16"),
               bt=torch.from_numpy(q1.block_tables).cuda(), ln=torch.from_numpy(q1.context_lens).cuda())
    q = to_device(q1.q, "bf16")
    a = pa.decode(q, dev["kc"], dev["vc"], dev["bt"], dev["ln"], scale=q1.scale, workspace=ws)
    b = pa.decode_multi(q.unsqueeze(1).contiguous(), dev["kc"], dev["vc"], dev["bt"], dev["ln"], scale=q1.scale,
                        workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b[:, 0].contiguous().view(torch.int16))


def test_multi_qwen_shape_sampled_rows():
    # speculative verify of 3 draft tokens (+1) on the Qwen-style batch: every row of 8 sequences
    inp = wl.make_decode_inputs("mq_qwen", context_lens=lambda r: r.integers(512, 4097, size=64), num_heads=28,
                                num_kv_heads=4, head_dim=128, block_size=16, dtype="bf16", num_blocks=20000, seed=0,
                                q_len=4)
    got = run_multi(inp)
    rng = np.random.default_rng(2)
    seqs = rng.choice(64, 8, replace=False)
    rows = [(int(b), t, h) for b in seqs for t in range(4) for h in range(28)]
    ref = oracle.decode_multi(inp.q, inp.key_cache, inp.value_cache, inp.block_tables, inp.context_lens, "bf16",
                              inp.scale, rows=rows)
    assert_decode_close(np.stack([got[b, t, h] for b, t, h in rows]), ref, "bf16")


@pytest.mark.parametrize("q_len", [2, 3, 4])
@pytest.mark.parametrize("lens,hkv", [((4096,), 1), ((0, 5000, 3), 2), ((700, 1, 0, 2049, 16, 17), 4)])
def test_row_split_schedule_cut_units(lens, hkv, q_len):
    # 9..32 rows per kv head take the persistent row-split wave.  With few pages against one wave of
    # CTAs a share holds one or two pages, so a unit spans up to hundreds of shares and the merge
    # folds more than 32 partial records into a row; empty and shorter-than-q_len contexts included.
    inp = mq_case("bf16", 128, 16, 7 * hkv, hkv, q_len, lens=lens, seed=len(lens) * 10 + q_len)
    plan = pa.decode_plan(inp.num_seqs, inp.num_heads, inp.num_kv_heads, 128, 16, inp.max_blocks_per_seq,
                          torch.bfloat16, q_len=q_len)
    assert plan.schedule == 2 and plan.grid_ctas > 0
    assert_decode_close(run_multi(inp).reshape(-1, 128), oracle_multi(inp).reshape(-1, 128), "bf16")
