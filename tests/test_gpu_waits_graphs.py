"""The lean schedule's merge: its bounded wait gives up cleanly, and a captured call replays.

* Give-up path: pa_diag_merge_timeout launches the merge alone, so the partial records it
  waits for are never published (a flag that nothing sets).  Its wait must end after the
  given bound with PA_ERR_TIMEOUT in the device error word, leave the output untouched,
  and leave the device usable: the next pa_decode must still match the oracle.
* Replay: pa_decode with a caller workspace captured in a CUDA graph reuses its epoch on
  every replay; the merge clears the flags it consumed, so each replay with new queries
  must match the oracle and a direct call bit for bit.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from paged_kv_cache_129_gb300 import workloads as wl
from helpers import assert_decode_close, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    pa.library()
    yield
    pa.check_error()


def lean_case(seed=3, lens=(1, 40, 300, 1000, 2049, 3000, 17, 700)):
    inp = wl.make_decode_inputs("lean", context_lens=list(lens), num_heads=28, num_kv_heads=4, head_dim=128,
                                block_size=16, dtype="bf16", pool_slack=0.3, seed=seed)
    plan = pa.decode_plan(inp.num_seqs, inp.num_heads, inp.num_kv_heads, inp.head_dim, inp.block_size,
                          inp.max_blocks_per_seq, torch.bfloat16)
    assert plan.schedule == 1, "these sizes must take the lean schedule"
    dev = dict(kc=to_device(inp.key_cache, "bf16"), vc=to_device(inp.value_cache, "bf16"),
               bt=torch.from_numpy(inp.block_tables).cuda(), lens=torch.from_numpy(inp.context_lens).cuda())
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    return inp, dev, ws


def bits(t):
    return t.view(torch.int16)


def test_merge_wait_gives_up_after_its_bound_and_the_device_stays_usable():
    inp, dev, ws = lean_case()
    q = to_device(inp.q, "bf16")
    # a normal call first: the workspace then holds published-and-cleared flags, as in use
    pa.decode(q, dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws)
    pa.check_error()
    sentinel = torch.full(q.shape, 0x7BAD, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    out = sentinel.clone()
    t0 = time.perf_counter()
    pa.diag_merge_timeout(out, dev["lens"], inp.num_kv_heads, inp.block_size, inp.max_blocks_per_seq, ws,
                          wait_limit_ns=1_000_000)
    with pytest.raises(pa.PAError) as err:
        pa.check_error()
    elapsed = time.perf_counter() - t0
    assert err.value.status == 8, err.value  # PA_ERR_TIMEOUT
    assert elapsed < 1.0, f"the 1 ms wait bound was not honoured ({elapsed:.3f} s)"
    assert torch.equal(bits(out), bits(sentinel)), "a merge that gave up wrote output"
    pa.check_error()  # the word was cleared by the read above
    # the device is still usable and correct
    got = pa.decode(q, dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws)
    pa.check_error()
    assert_decode_close(to_f64(got), oracle.decode_inputs(inp), "bf16")


def test_diag_merge_refuses_plans_without_the_lean_schedule():
    # 256 MHA sequences: more units than consumer warps, so pa_decode takes the partitioned grid
    inp = wl.make_decode_inputs("grid", context_lens=[64] * 256, num_heads=32, num_kv_heads=32, head_dim=128,
                                block_size=16, dtype="f16", pool_slack=0.1, seed=1)
    out = torch.zeros(256, 32, 128, dtype=torch.float16, device="cuda")
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    lens = torch.from_numpy(inp.context_lens).cuda()
    with pytest.raises(pa.PAError) as err:
        pa.diag_merge_timeout(out, lens, 32, 16, inp.max_blocks_per_seq, ws, wait_limit_ns=1_000_000)
    assert err.value.status == 1


def test_captured_lean_call_replays_with_new_queries():
    inp, dev, ws = lean_case(seed=5)
    q_static = to_device(inp.q, "bf16")
    out_static = torch.empty_like(q_static)
    pa.decode(q_static, dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws,
              out=out_static)  # set-up before capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.decode(q_static, dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws,
                  out=out_static)
    for seed in (11, 12, 13):
        qn = wl.make_decode_inputs("lean", context_lens=list(inp.context_lens), num_heads=28, num_kv_heads=4,
                                   head_dim=128, block_size=16, dtype="bf16", pool_slack=0.3, seed=seed).q
        q_static.copy_(to_device(qn, "bf16"))
        graph.replay()
        torch.cuda.synchronize()
        pa.check_error()
        case = inp
        case_q, case.q = case.q, qn
        ref = oracle.decode_inputs(case)
        case.q = case_q
        assert_decode_close(to_f64(out_static), ref, "bf16")
        direct = pa.decode(q_static, dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(bits(out_static), bits(direct))
