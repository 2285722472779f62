"""pa_decode_static_scratch: pa_decode with the library's built-in scratch.

Each case runs two calls in a row through the static-scratch entry point
(different queries, so the second call cannot lean on what the first left in
the scratch).  Both outputs are checked against the CPU oracle at the decode
tolerance, and must be bit-identical to pa_decode given a caller-allocated
workspace of the same size (the same plan, so the same arithmetic in the same
order).  The file runs last on purpose, after every other GPU test has used
the library, and also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from paged_kv_cache_129_gb300 import workloads as wl
from helpers import TORCH_DTYPE, assert_decode_close, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    yield
    pa.check_error()


def upload(inp):
    return dict(kc=to_device(inp.key_cache, inp.dtype), vc=to_device(inp.value_cache, inp.dtype),
                bt=torch.from_numpy(inp.block_tables).cuda(), lens=torch.from_numpy(inp.context_lens).cuda())


def need_bytes(inp):
    return pa.decode_workspace_size(inp.num_seqs, inp.num_heads, inp.num_kv_heads, inp.head_dim, inp.block_size,
                                    inp.max_blocks_per_seq, TORCH_DTYPE[inp.dtype])


def with_workspace(q, dev, inp, raw=False):
    ws_bytes = need_bytes(inp)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = pa.decode(q, dev["kc"], dev["vc"], dev["bt"], dev["lens"], scale=inp.scale, workspace=ws)
    torch.cuda.synchronize()
    pa.check_error()
    return out if raw else to_f64(out)


def bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


def alloc_count():
    return torch.cuda.memory_stats().get("allocation.all.allocated", 0)


CASES = {
    # lean schedule with merges: few sequences, GQA 7, ragged lengths (tails of 1..15 tokens)
    "lean_bf16_gqa": dict(num_seqs=12, num_heads=28, num_kv_heads=4, head_dim=128, block_size=16, dtype="bf16",
                          lens=(1, 17, 300, 1000, 2049, 4095, 33, 15, 16, 777, 3000, 129)),
    # CUDA-core kernel, fp32, MHA, block size 32
    "lean_f32_mha": dict(num_seqs=5, num_heads=4, num_kv_heads=4, head_dim=64, block_size=32, dtype="f32",
                         lens=(0, 1, 95, 640, 2000)),
    # enough (sequence, kv head) units for one whole-context pass: no scratch at all
    "single_pass_f16": dict(num_seqs=128, num_heads=32, num_kv_heads=32, head_dim=128, block_size=16, dtype="f16",
                            lens=None),
}


def make_case(spec, seed):
    lens = spec["lens"]
    if lens is None:
        lens = np.random.default_rng(seed).integers(16, 200, spec["num_seqs"])
    return wl.make_decode_inputs("static_scratch", num_heads=spec["num_heads"], num_kv_heads=spec["num_kv_heads"],
                                 head_dim=spec["head_dim"], block_size=spec["block_size"], dtype=spec["dtype"],
                                 context_lens=np.asarray(lens), seed=seed)


@pytest.mark.parametrize("name", list(CASES))
def test_two_calls_match_pa_decode(name):
    spec = CASES[name]
    inp = make_case(spec, seed=101)
    if name == "single_pass_f16":
        assert need_bytes(inp) == 0
    else:
        assert 0 < need_bytes(inp) <= pa.STATIC_SCRATCH_BYTES
    dev = upload(inp)
    q1 = to_device(inp.q, inp.dtype)
    q2 = to_device(make_case(spec, seed=202).q, inp.dtype)
    out1, out2 = torch.empty_like(q1), torch.empty_like(q2)
    # the first call does the setup; after it, the calls allocate nothing through torch
    pa.decode_static_scratch(q1, dev["kc"], dev["vc"], dev["bt"], dev["lens"], out1, scale=inp.scale)
    torch.cuda.synchronize()
    before = alloc_count()
    pa.decode_static_scratch(q1, dev["kc"], dev["vc"], dev["bt"], dev["lens"], out1, scale=inp.scale)
    pa.decode_static_scratch(q2, dev["kc"], dev["vc"], dev["bt"], dev["lens"], out2, scale=inp.scale)
    torch.cuda.synchronize()
    assert alloc_count() == before
    pa.check_error()
    inp2 = make_case(spec, seed=202)
    for out, q, case in ((out1, q1, inp), (out2, q2, inp2)):
        # against the CPU oracle, at the decode tolerance
        case.key_cache, case.value_cache, case.block_tables = inp.key_cache, inp.value_cache, inp.block_tables
        case.context_lens = inp.context_lens
        assert_decode_close(to_f64(out), oracle.decode_inputs(case), inp.dtype)
        # and bit for bit what pa_decode computes with a workspace of the same size (the same plan)
        assert torch.equal(bits(out), bits(with_workspace(q, dev, inp, raw=True)))


def test_sizes_beyond_the_static_scratch_are_refused():
    # head_dim 256 keeps one 8-head record of 8 KB per consumer warp slot; on a
    # 152-SM GB300 the lean plan needs ~20 MB, more than the 16 MB built in.
    inp = wl.make_decode_inputs("static_scratch_d256", num_heads=16, num_kv_heads=2, head_dim=256, block_size=16, dtype="bf16",
                                context_lens=np.array([100, 3000]), seed=7)
    need = need_bytes(inp)
    if need <= pa.STATIC_SCRATCH_BYTES:
        pytest.skip(f"this device's plan for head_dim 256 needs only {need} bytes")
    dev = upload(inp)
    q = to_device(inp.q, inp.dtype)
    out = torch.zeros_like(q)
    with pytest.raises(pa.PAError) as err:
        pa.decode_static_scratch(q, dev["kc"], dev["vc"], dev["bt"], dev["lens"], out, scale=inp.scale)
    assert err.value.status == 2 and str(need) in str(err.value) and "PA_STATIC_SCRATCH_BYTES" in str(err.value)
    torch.cuda.synchronize()
    assert not out.any()  # nothing was launched
    # the same sizes through pa_decode with a workspace still work
    got = with_workspace(q, dev, inp)
    assert np.isfinite(got).all()


def test_zero_sequences_is_a_no_op():
    lib = pa.library()
    assert lib.pa_decode_static_scratch(None, None, None, None, None, None, 0, 8, 2, 128, 16, 1, 1,
                                        ctypes.c_float(1.0), 2, None) == 0
