"""The lean decode's early set-up: read before the dependency wait, checked after it.

The lean decode reads the context lengths and each warp's first block-table rows before it
waits for the previous kernel in the stream, issues its first page loads from them the
moment the wait returns, and re-reads both to check them; a CTA whose early reads differ
discards those pages and sets up again.  Two kinds of test:

* pa_diag_force_restart makes every CTA take that second path: parity cases of every lean
  consumer (16-bit tensor-core, CUDA-core fp32, append mode, FP8, multi-query) must still
  match the oracle.
* The previous kernel really changes the inputs: pa_apply_table_deltas rewrites block-table
  rows right before a pa_decode on the same stream, alternating between two tables whose
  pages hold different data; every output must match the oracle for the table it was given.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from paged_kv_cache_129_gb300 import workloads as wl
from helpers import assert_decode_close, to_device, to_f64
from test_gpu_append import test_append_matches_oracle_and_unfused_path as _append_case
from test_gpu_fp8 import test_decode_fp8_append_matches_write_then_decode as _fp8_append_case
from test_gpu_fp8 import test_decode_fp8_matches_oracle as _fp8_case
from test_gpu_kernels import test_decode_matches_oracle as _decode_case
from test_gpu_kernels import test_tiny_workload as _tiny_case
from test_gpu_multi import test_multi_matches_oracle as _multi_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    pa.library()
    yield
    pa.diag_force_restart(False)
    pa.check_error()


@pytest.fixture
def restart():
    pa.diag_force_restart(True)
    try:
        yield
    finally:
        pa.diag_force_restart(False)


@pytest.mark.parametrize("dtype,d,bs,hq,hkv,kernel", [
    ("bf16", 128, 16, 28, 4, "mma"), ("f16", 128, 32, 32, 32, "mma"), ("bf16", 256, 16, 8, 2, "mma"),
    ("f16", 128, 16, 32, 2, "mma"), ("bf16", 128, 16, 28, 4, "simt"), ("f32", 64, 16, 4, 2, "simt")])
def test_restarted_setup_decode(restart, dtype, d, bs, hq, hkv, kernel):
    _decode_case(dtype, d, bs, hq, hkv, kernel, 0)


def test_restarted_setup_tiny(restart):
    _tiny_case(0)


@pytest.mark.parametrize("dtype,d,bs,hq,hkv,kernel", [("bf16", 128, 16, 28, 4, "mma"), ("f32", 128, 16, 28, 4, "simt")])
def test_restarted_setup_append(restart, dtype, d, bs, hq, hkv, kernel):
    _append_case(dtype, d, bs, hq, hkv, kernel, 0)


@pytest.mark.parametrize("bs,hq,hkv", [(16, 28, 4), (32, 8, 8)])
def test_restarted_setup_fp8(restart, bs, hq, hkv):
    _fp8_case("bf16", bs, hq, hkv)


def test_restarted_setup_fp8_append(restart):
    _fp8_append_case("bf16", 16, "interleaved", 28, 4)


def test_restarted_setup_multi_query(restart):
    _multi_case("bf16", 128, 16, 28, 4, "mma", 4, 0)
    from test_gpu_multi import test_multi_many_rows_per_kv_head as _many_rows
    _many_rows(9)


def test_tables_rewritten_by_the_previous_kernel():
    # Two tables over one pool for the same lengths (disjoint physical blocks, different data).
    # Each step rewrites every entry of the device table with pa_apply_table_deltas and decodes
    # at once on the same stream: the decode's early reads may see the old table, its checked
    # reads see the new one, and the output must be the new table's.
    lens = [1, 40, 300, 1000, 2049, 3000, 17, 700]
    inp = wl.make_decode_inputs("two_tables", context_lens=lens, num_heads=28, num_kv_heads=4, head_dim=128,
                                block_size=16, dtype="bf16", pool_slack=1.2, seed=9)
    need = [(n + 15) // 16 for n in lens]
    used = set(int(x) for b in range(len(lens)) for x in inp.block_tables[b, :need[b]])
    spare = np.array(sorted(set(range(inp.num_blocks)) - used), dtype=np.int32)
    spare = np.random.default_rng(1).permutation(spare)
    tab_a = inp.block_tables.copy()
    tab_b = np.full_like(tab_a, -1)
    cur = 0
    for b, k in enumerate(need):
        tab_b[b, :k] = spare[cur:cur + k]
        cur += k
    plan = pa.decode_plan(inp.num_seqs, 28, 4, 128, 16, tab_a.shape[1], torch.bfloat16)
    assert plan.schedule == 1
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    kc, vc = to_device(inp.key_cache, "bf16"), to_device(inp.value_cache, "bf16")
    q, lens_d = to_device(inp.q, "bf16"), torch.from_numpy(inp.context_lens).cuda()

    def deltas(tab):
        rows = [(b, j, int(tab[b, j])) for b in range(len(lens)) for j in range(need[b])]
        return torch.tensor(rows, dtype=torch.int32).cuda()

    d_a, d_b = deltas(tab_a), deltas(tab_b)
    dev_tab = torch.from_numpy(tab_a).cuda()
    outs, which = [], []
    torch.cuda.synchronize()
    for step in range(8):
        use_b = step % 2 == 0
        pa.apply_table_deltas(dev_tab, d_b if use_b else d_a)
        outs.append(pa.decode(q, kc, vc, dev_tab, lens_d, scale=inp.scale, workspace=ws))
        which.append(use_b)
    torch.cuda.synchronize()
    pa.check_error()
    refs = {}
    for use_b in (False, True):
        inp.block_tables = tab_b if use_b else tab_a
        refs[use_b] = oracle.decode_inputs(inp)
    for out, use_b in zip(outs, which):
        assert_decode_close(to_f64(out), refs[use_b], "bf16")
