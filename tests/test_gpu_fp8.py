"""GPU parity of the FP8 (E4M3) KV-cache path against the oracle.

* pa_write_kv_fp8: bit-exact against the oracle's quantiser for bf16 / f16 / f32 sources,
  saturating and NaN inputs, padding slots, a bad slot flagged;
* pa_decode_fp8: within the bf16/f16 tolerance (|err| <= 2e-2 + 1e-2 |ref|) of the oracle's
  fp64 attention over the same codes and scales, on ragged contexts (L = 0, 1, 15, 16, 17, ...)
  at block sizes 16 and 32, NaN codes in the slots past each context, scales that differ per
  (block, kv head), and queries of magnitudes far outside f16's range;
* the Qwen-shaped layer at full size (the shape the benchmark times): the caches written by
  the GPU writer equal the oracle's byte for byte, and sampled output rows match the oracle;
* pa_decode_fp8_append (the new token quantised at position L - 1 inside the decode): the
  caches equal the oracle's writer at those slots byte for byte, the output is bit-identical to
  pa_write_kv_fp8 + pa_decode_fp8 and within tolerance of the oracle, for both layouts, block
  sizes 16 and 32, GQA groups that take one and two head chunks, and at full Qwen size.
"""
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
    pa.library()
    yield
    pa.check_error()


def _src(rng, shape, dtype, mult=1.0):
    x = (rng.standard_normal(shape) * mult).astype(np.float32)
    return wl.cast_from_f32(x, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_write_kv_fp8_bit_exact(dtype):
    rng = np.random.default_rng(11)
    nb, hkv, bs, d, T = 9, 4, 16, 128, 40
    kc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    vc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    ks = rng.uniform(0.004, 0.05, (nb, hkv)).astype(np.float32)
    vs = rng.uniform(0.004, 0.05, (nb, hkv)).astype(np.float32)
    key = _src(rng, (T, hkv, d), dtype, 3.0)
    val = _src(rng, (T, hkv, d), dtype, 3.0)
    if dtype == "f32":
        key[0, 0, :4] = [1e6, -1e6, np.nan, 1e-30]  # saturating, NaN and tiny inputs
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int64)
    slots[::9] = -1
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    pa.write_kv_fp8(to_device(key, dtype), to_device(val, dtype), dk, dv, torch.from_numpy(ks).cuda(),
                    torch.from_numpy(vs).cuda(), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert oracle.write_kv_fp8(key, val, dtype, kc, vc, ks, vs, slots) == oracle.OK
    assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
    pa.check_error()


def test_write_kv_fp8_flags_a_bad_slot():
    nb, hkv, bs, d = 2, 1, 16, 128
    dk = torch.zeros(nb, hkv, bs, d, dtype=torch.uint8, device="cuda")
    dv = torch.zeros_like(dk)
    one = torch.ones(nb, hkv, device="cuda")
    rows = torch.ones(2, hkv, d, device="cuda")
    pa.write_kv_fp8(rows, rows, dk, dv, one, one, torch.tensor([3, nb * bs], dtype=torch.int64, device="cuda"))
    with pytest.raises(pa.PAError) as e:
        pa.check_error()
    assert e.value.status == 6
    assert int((dk != 0).sum()) == d  # slot 3 written with code(1.0) = 0x38, nothing else
    assert int(dk[0, 0, 3, 0]) == 0x38


def _case(seed, lens, hq, hkv, bs, dtype, q_mult=1.0, slack=2):
    rng = np.random.default_rng(seed)
    d = 128
    lens = np.asarray(lens, np.int32)
    nblk = (lens + bs - 1) // bs
    nb = int(nblk.sum()) + slack
    perm = rng.permutation(nb)
    width = max(1, int(nblk.max()))
    bt = np.full((len(lens), width), -1, np.int32)
    k = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[k:k + n]
        k += n
    kc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    vc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x3A  # no NaN codes inside the contexts ...
    vc[(vc & 0x7F) == 0x7F] = 0x3B
    for b, L in enumerate(lens):  # ... but NaN codes in every slot past a context
        if L % bs:
            blk = bt[b, L // bs]
            kc[blk, :, L % bs:] = 0x7F
            vc[blk, :, L % bs:] = 0xFF
    ks = rng.uniform(0.002, 0.02, (nb, hkv)).astype(np.float32)
    vs = rng.uniform(0.002, 0.02, (nb, hkv)).astype(np.float32)
    q = _src(rng, (len(lens), hq, d), dtype, q_mult)
    return q, kc, vc, ks, vs, bt, lens


def _run(q, kc, vc, ks, vs, bt, lens, dtype):
    out = pa.decode_fp8(to_device(q, dtype), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                        torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(), torch.from_numpy(bt).cuda(),
                        torch.from_numpy(lens).cuda())
    torch.cuda.synchronize()
    return to_f64(out)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("hq,hkv", [(28, 4), (8, 8), (32, 8)])
def test_decode_fp8_matches_oracle(dtype, bs, hq, hkv):
    lens = [0, 1, 15, 16, 17, 33, 250, 1000, 2047, 64]
    q, kc, vc, ks, vs, bt, lens = _case(hq * bs + hkv, lens, hq, hkv, bs, dtype)
    got = _run(q, kc, vc, ks, vs, bt, lens, dtype)
    ref = oracle.decode_fp8(q, dtype, kc, vc, ks, vs, bt, lens, 1 / np.sqrt(128))
    assert_decode_close(got, ref, dtype)
    assert np.all(got[0] == 0)  # empty context: a zero row
    pa.check_error()


@pytest.mark.parametrize("dtype,q_mult", [("bf16", 3e5), ("bf16", 1e-6), ("f16", 2000.0)])
def test_decode_fp8_queries_outside_f16_range(dtype, q_mult):
    # the query row is scaled by a power of two into f16 range: exact for any magnitude
    q, kc, vc, ks, vs, bt, lens = _case(7, [40, 300, 5], 28, 4, 16, dtype, q_mult=q_mult)
    scale = 1 / np.sqrt(128)
    got = _run(q, kc, vc, ks, vs, bt, lens, dtype)
    ref = oracle.decode_fp8(q, dtype, kc, vc, ks, vs, bt, lens, scale)
    assert_decode_close(got, ref, dtype)


def test_qwen_layer_fp8_full_size():
    """The Qwen-shaped layer (batch 64, 28/4 heads, d 128, bs 16, L ~ U[512, 4096], pool 20000) with
    per-(block, head) scales from the block's source values: the caches the GPU writer quantises equal
    the oracle's byte for byte; sampled output rows match the oracle."""
    inp = wl.qwen_gqa(0)
    ks, vs = wl.fp8_scales(inp.key_cache, inp.dtype), wl.fp8_scales(inp.value_cache, inp.dtype)
    nb, hkv, bs, d = inp.key_cache.shape
    # quantise the whole pool: every slot written once through the writer
    slots = np.arange(nb * bs, dtype=np.int64)
    src_k = np.ascontiguousarray(inp.key_cache.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    src_v = np.ascontiguousarray(inp.value_cache.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    dk = torch.empty(nb, hkv, bs, d, dtype=torch.uint8, device="cuda")
    dv = torch.empty_like(dk)
    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    pa.write_kv_fp8(to_device(src_k, inp.dtype), to_device(src_v, inp.dtype), dk, dv, dks, dvs,
                    torch.from_numpy(slots).cuda())
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = np.zeros_like(kc)
    assert oracle.write_kv_fp8(src_k, src_v, inp.dtype, kc, vc, ks, vs, slots) == oracle.OK
    torch.cuda.synchronize()
    assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
    out = pa.decode_fp8(to_device(inp.q, inp.dtype), dk, dv, dks, dvs, torch.from_numpy(inp.block_tables).cuda(),
                        torch.from_numpy(inp.context_lens).cuda())
    torch.cuda.synchronize()
    got = to_f64(out)
    rng = np.random.default_rng(1)
    rows = [(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 48), rng.integers(0, 28, 48))]
    ref = oracle.decode_fp8(inp.q, inp.dtype, kc, vc, ks, vs, inp.block_tables, inp.context_lens, inp.scale, rows)
    assert_decode_close(np.stack([got[b, h] for b, h in rows]), ref, inp.dtype)
    pa.check_error()


@pytest.mark.parametrize("fp8_write", ["separate", "fused"])
def test_stepper_fp8_matches_direct_calls(fp8_write):
    """pa.DecodeStepper over FP8 caches (new tokens quantised at their slots then the FP8 decode, or the
    fused pa_decode_fp8_append; block tables kept by deltas) gives the same bytes as the direct calls."""
    rng = np.random.default_rng(21)
    B, hq, hkv, bs, d, steps = 6, 28, 4, 16, 128, 5
    lens = rng.integers(1, 300, B).astype(np.int32)
    nblk = (lens + bs - 1) // bs
    nb = int(nblk.sum()) + 4
    perm = rng.permutation(nb)
    width = int(nblk.max())
    bt = np.full((B, width), -1, np.int32)
    k = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[k:k + n]
        k += n
    slots = np.array([bt[b, (L - 1) // bs] * bs + (L - 1) % bs for b, L in enumerate(lens)], np.int64)
    kc = torch.from_numpy(rng.integers(0, 0x7E, (nb, hkv, bs, d), dtype=np.uint8)).cuda()
    vc = torch.from_numpy(rng.integers(0, 0x7E, (nb, hkv, bs, d), dtype=np.uint8)).cuda()
    ks = torch.from_numpy(rng.uniform(0.005, 0.02, (nb, hkv)).astype(np.float32)).cuda()
    vs = torch.from_numpy(rng.uniform(0.005, 0.02, (nb, hkv)).astype(np.float32)).cuda()
    kc_ref, vc_ref = kc.clone(), vc.clone()
    stepper = pa.DecodeStepper(kc, vc, B, hq, width, append=True, tables="deltas", k_scale=ks, v_scale=vs,
                               query_dtype=torch.bfloat16, fp8_write=fp8_write)
    deltas = np.array([(r, j, bt[r, j]) for r in range(B) for j in range(nblk[r])], np.int32)
    got, refs = [], []
    ws = torch.empty(max(pa.decode_fp8_workspace_size(B, hq, hkv, d, bs, width, torch.bfloat16), 256),
                     dtype=torch.uint8, device="cuda")
    for i in range(steps):
        if i >= stepper.slots:
            got.append(stepper.result(i - stepper.slots).clone())
        q = torch.randn(B, hq, d).to(torch.bfloat16)
        nk = torch.randn(B, hkv, d).to(torch.bfloat16)
        nv = torch.randn(B, hkv, d).to(torch.bfloat16)
        v = stepper.inputs(i)
        v.query.copy_(q)
        v.new_key.copy_(nk)
        v.new_value.copy_(nv)
        if fp8_write == "separate":
            v.slots.copy_(torch.from_numpy(slots))
        else:
            assert not hasattr(v, "slots")  # the fused step derives the slots from the tables
        v.context_lens.copy_(torch.from_numpy(lens))
        n = len(deltas) if i == 0 else 0
        v.deltas.numpy()[:n] = deltas[:n]
        stepper.launch(i, num_deltas=n)
        dbt, dl = torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda()
        if fp8_write == "separate":
            pa.write_kv_fp8(nk.cuda(), nv.cuda(), kc_ref, vc_ref, ks, vs, torch.from_numpy(slots).cuda())
            refs.append(pa.decode_fp8(q.cuda(), kc_ref, vc_ref, ks, vs, dbt, dl, workspace=ws))
        else:
            refs.append(pa.decode_fp8_append(q.cuda(), nk.cuda(), nv.cuda(), kc_ref, vc_ref, ks, vs, dbt, dl,
                                             workspace=ws))
    for i in range(steps - stepper.slots, steps):
        got.append(stepper.result(i).clone())
    torch.cuda.synchronize()
    pa.check_error()
    for i in range(steps):
        assert torch.equal(got[i].view(torch.int16), refs[i].cpu().view(torch.int16)), f"step {i}"
    assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref)


@pytest.mark.parametrize("bs", [16, 32])
def test_interleaved_layout_matches_separate_caches(bs):
    """The interleaved FP8 layout ([N, H_kv, 2, bs, d]: K rows then V rows of each (block, kv head), one
    copy per page): the writer stores the same codes as into separate caches (bit-exact against the oracle),
    and the decode gives the same bits as over separate caches, within tolerance of the oracle."""
    rng = np.random.default_rng(bs)
    hq, hkv, d = 28, 4, 128
    q, kc, vc, ks, vs, bt, lens = _case(40 + bs, [1, 17, 300, 1000, 64, 0], hq, hkv, bs, "bf16")
    nb = kc.shape[0]
    # the writer: every slot of the pool from bf16 sources
    src_k = _src(rng, (nb * bs, hkv, d), "bf16", 2.0)
    src_v = _src(rng, (nb * bs, hkv, d), "bf16", 2.0)
    slots = np.arange(nb * bs, dtype=np.int64)
    kv = torch.empty(nb, hkv, 2, bs, d, dtype=torch.uint8, device="cuda")
    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    pa.write_kv_fp8(to_device(src_k, "bf16"), to_device(src_v, "bf16"), kv, None, dks, dvs,
                    torch.from_numpy(slots).cuda())
    exp_k, exp_v = np.zeros_like(kc), np.zeros_like(vc)
    assert oracle.write_kv_fp8(src_k, src_v, "bf16", exp_k, exp_v, ks, vs, slots) == oracle.OK
    torch.cuda.synchronize()
    got = kv.cpu().numpy()
    assert np.array_equal(got[:, :, 0], exp_k) and np.array_equal(got[:, :, 1], exp_v)
    # the decode over the interleaved layout vs separate caches and the oracle
    kv2 = torch.from_numpy(np.ascontiguousarray(np.stack([kc, vc], axis=2))).cuda()
    dq, dbt, dl = to_device(q, "bf16"), torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda()
    inter = pa.decode_fp8(dq, kv2, None, dks, dvs, dbt, dl)
    sep = pa.decode_fp8(dq, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(), dks, dvs, dbt, dl)
    torch.cuda.synchronize()
    assert torch.equal(inter.view(torch.int16), sep.view(torch.int16))
    ref = oracle.decode_fp8(q, "bf16", kc, vc, ks, vs, bt, lens, 1 / np.sqrt(d))
    assert_decode_close(to_f64(inter), ref, "bf16")
    pa.check_error()


@pytest.mark.parametrize("layout", ["separate", "interleaved"])
def test_fp8_copy_and_swap_bit_exact(layout):
    """Copy-on-write block copies and swaps of FP8 caches (one-byte elements; the interleaved layout copies
    each [H_kv, 2, bs, d] record whole) equal the oracle's byte copies."""
    rng = np.random.default_rng(31)
    nb, hkv, bs, d = 12, 4, 16, 128
    shape = (nb, hkv, 2, bs, d) if layout == "interleaved" else (nb, hkv, bs, d)
    kc = rng.integers(0, 256, shape, dtype=np.uint8)
    vc = None if layout == "interleaved" else rng.integers(0, 256, shape, dtype=np.uint8)
    pairs = np.array([[1, 7], [3, 9], [0, 11]], np.int64)
    dk = torch.from_numpy(kc).cuda()
    dv = torch.from_numpy(vc).cuda() if vc is not None else None
    pa.copy_blocks(dk, dv, torch.from_numpy(pairs).cuda())
    exp_k = kc.copy()
    exp_v = vc.copy() if vc is not None else exp_k
    assert oracle.copy_blocks(exp_k, exp_v, pairs) == oracle.OK
    torch.cuda.synchronize()
    assert np.array_equal(dk.cpu().numpy(), exp_k)
    if vc is not None:
        assert np.array_equal(dv.cpu().numpy(), exp_v)
    # swap out to page-locked host memory and back into other blocks
    hk = torch.zeros((5,) + shape[1:], dtype=torch.uint8).pin_memory()
    hv = torch.zeros_like(hk).pin_memory() if vc is not None else None
    out_pairs = np.array([[7, 0], [9, 3], [2, 4]], np.int64)
    pa.swap_blocks(hk, hv, dk, dv, torch.from_numpy(out_pairs).cuda())
    in_pairs = np.array([[0, 5], [3, 6], [4, 8]], np.int64)
    in_host = torch.from_numpy(in_pairs).pin_memory()
    pa.swap_blocks(dk, dv, hk, hv, in_host)
    torch.cuda.synchronize()
    h_exp_k = np.zeros((5,) + shape[1:], np.uint8)
    h_exp_v = np.zeros_like(h_exp_k) if vc is not None else h_exp_k
    assert oracle.swap_blocks(h_exp_k, h_exp_v, exp_k, exp_v, out_pairs) == oracle.OK
    assert oracle.swap_blocks(exp_k, exp_v, h_exp_k, h_exp_v, in_pairs) == oracle.OK
    assert np.array_equal(hk.numpy(), h_exp_k) and np.array_equal(dk.cpu().numpy(), exp_k)
    if vc is not None:
        assert np.array_equal(hv.numpy(), h_exp_v) and np.array_equal(dv.cpu().numpy(), exp_v)
    pa.check_error()


def _new_token_slots(bt, lens, bs):
    """Slots of positions L - 1 through the block tables (-1 for an empty context)."""
    return np.array([bt[b, (L - 1) // bs] * bs + (L - 1) % bs if L >= 1 else -1 for b, L in enumerate(lens)],
                    np.int64)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("layout", ["separate", "interleaved"])
@pytest.mark.parametrize("hq,hkv", [(28, 4), (8, 8), (32, 2)])
def test_decode_fp8_append_matches_write_then_decode(dtype, bs, layout, hq, hkv):
    """pa_decode_fp8_append: the new token of each sequence quantised with its block's scales at position
    L - 1 (the first, a middle and the last row of a page; L = 0 writes nothing), then attended.  Group 16
    (32 / 2 heads) splits each kv head into two head chunks, which patch the staged page alike while
    only the first stores it."""
    d = 128
    lens = [0, 1, 15, 16, 17, 33, 250, 1000, 64, 2]
    q, kc, vc, ks, vs, bt, lens = _case(hq * bs + hkv + 5, lens, hq, hkv, bs, dtype)
    rng = np.random.default_rng(hq + bs)
    nk = _src(rng, (len(lens), hkv, d), dtype, 1.5)  # |x| / scale spans normal codes and saturation
    nv = _src(rng, (len(lens), hkv, d), dtype, 1.5)
    slots = _new_token_slots(bt, lens, bs)
    ek, ev = kc.copy(), vc.copy()
    assert oracle.write_kv_fp8(nk, nv, dtype, ek, ev, ks, vs, slots) == oracle.OK
    ref = oracle.decode_fp8(q, dtype, ek, ev, ks, vs, bt, lens, 1 / np.sqrt(d))

    def caches():
        if layout == "interleaved":
            return torch.from_numpy(np.ascontiguousarray(np.stack([kc, vc], axis=2))).cuda(), None
        return torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()

    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    dq, dbt, dl = to_device(q, dtype), torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda()
    dnk, dnv = to_device(nk, dtype), to_device(nv, dtype)
    ws = torch.empty(max(pa.decode_fp8_workspace_size(len(lens), hq, hkv, d, bs, bt.shape[1], TORCH_DTYPE[dtype]),
                         256), dtype=torch.uint8, device="cuda")
    fk, fv = caches()
    fused = pa.decode_fp8_append(dq, dnk, dnv, fk, fv, dks, dvs, dbt, dl, workspace=ws)
    uk, uv = caches()
    pa.write_kv_fp8(dnk, dnv, uk, uv, dks, dvs, torch.from_numpy(slots).cuda())
    unfused = pa.decode_fp8(dq, uk, uv, dks, dvs, dbt, dl, workspace=ws)
    torch.cuda.synchronize()
    if layout == "interleaved":
        assert np.array_equal(fk.cpu().numpy(), np.stack([ek, ev], axis=2))
    else:
        assert np.array_equal(fk.cpu().numpy(), ek) and np.array_equal(fv.cpu().numpy(), ev)
    assert torch.equal(fused.view(torch.int16), unfused.view(torch.int16))
    got = to_f64(fused)
    assert_decode_close(got, ref, dtype)
    assert np.all(got[0] == 0)
    pa.check_error()


def test_qwen_layer_fp8_append_full_size():
    """The step the benchmark times for the FP8 Qwen-shaped layer (batch 64, 28/4 heads, d 128, bs 16,
    L ~ U[512, 4096], pool 20000, interleaved layout): after pa_decode_fp8_append the whole pool equals the
    oracle's (its quantised pool plus the new tokens at positions L - 1) byte for byte, and sampled output
    rows match the oracle's decode over it."""
    inp = wl.qwen_gqa(0)
    ks, vs = wl.fp8_scales(inp.key_cache, inp.dtype), wl.fp8_scales(inp.value_cache, inp.dtype)
    nb, hkv, bs, d = inp.key_cache.shape
    slots = np.arange(nb * bs, dtype=np.int64)
    src_k = np.ascontiguousarray(inp.key_cache.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    src_v = np.ascontiguousarray(inp.value_cache.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    kv = torch.empty(nb, hkv, 2, bs, d, dtype=torch.uint8, device="cuda")
    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    pa.write_kv_fp8(to_device(src_k, inp.dtype), to_device(src_v, inp.dtype), kv, None, dks, dvs,
                    torch.from_numpy(slots).cuda())
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = np.zeros_like(kc)
    assert oracle.write_kv_fp8(src_k, src_v, inp.dtype, kc, vc, ks, vs, slots) == oracle.OK
    new_slots = _new_token_slots(inp.block_tables, inp.context_lens, bs)
    assert oracle.write_kv_fp8(inp.new_key, inp.new_value, inp.dtype, kc, vc, ks, vs, new_slots) == oracle.OK
    out = pa.decode_fp8_append(to_device(inp.q, inp.dtype), to_device(inp.new_key, inp.dtype),
                               to_device(inp.new_value, inp.dtype), kv, None, dks, dvs,
                               torch.from_numpy(inp.block_tables).cuda(), torch.from_numpy(inp.context_lens).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(kv.cpu().numpy(), np.stack([kc, vc], axis=2))
    got = to_f64(out)
    rng = np.random.default_rng(2)
    rows = [(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 48), rng.integers(0, 28, 48))]
    ref = oracle.decode_fp8(inp.q, inp.dtype, kc, vc, ks, vs, inp.block_tables, inp.context_lens, inp.scale, rows)
    assert_decode_close(np.stack([got[b, h] for b, h in rows]), ref, inp.dtype)
    pa.check_error()


@pytest.mark.parametrize("layout", ["separate", "interleaved"])
def test_decode_fp8_more_units_than_warps(layout):
    """More (sequence, kv head) units than the lean decode has consumer warps (300 x 8 = 2400 units
    against 152 SMs x 3 CTAs x 4 warps): the merge then runs one CTA per boundary between two warps'
    shares, merging each cut unit once; every output row matches the oracle."""
    rng = np.random.default_rng(77)
    lens = rng.integers(1, 200, 300).astype(np.int32)
    lens[::37] = 16  # units that end exactly on a page edge
    q, kc, vc, ks, vs, bt, lens = _case(78, lens, 8, 8, 16, "f16")
    assert len(lens) * 8 > torch.cuda.get_device_properties(0).multi_processor_count * 3 * 4
    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    dq, dbt, dl = to_device(q, "f16"), torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda()
    if layout == "interleaved":
        got = pa.decode_fp8(dq, torch.from_numpy(np.ascontiguousarray(np.stack([kc, vc], axis=2))).cuda(), None, dks,
                            dvs, dbt, dl)
    else:
        got = pa.decode_fp8(dq, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(), dks, dvs, dbt, dl)
    torch.cuda.synchronize()
    ref = oracle.decode_fp8(q, "f16", kc, vc, ks, vs, bt, lens, 1 / np.sqrt(128))
    assert_decode_close(to_f64(got), ref, "f16")
    pa.check_error()
