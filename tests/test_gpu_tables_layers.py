"""GPU parity of the multi-layer write (pa_write_kv_layers) and of the block-table
delta path (pa_pool_table_deltas + pa_apply_table_deltas) against the oracle: bit-exact.

* multi-layer write: every layer's caches equal the oracle's per-layer write, for
  several dtypes, vector widths and layer counts (1 .. PA_MAX_LAYERS), padding
  slots skipped and a bad slot flagged;
* deltas: device- and pinned-host deltas applied equal the oracle's application,
  out-of-range entries flagged; a device table kept current only by delta exports
  over random pool operations equals the full export, and decoding through it
  gives the same bits as decoding through the full export.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_129_gb300 as pa
from helpers import TORCH_DTYPE, to_device, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; the CUDA path has no fallback"
    pa.build()
    pa.library()
    yield
    pa.check_error()


def _bits(rng, shape, dtype):
    if dtype == "f32":
        return rng.standard_normal(shape).astype(np.float32)
    if dtype == "f16":
        return rng.standard_normal(shape).astype(np.float16)
    return rng.integers(0, 2**16, shape, dtype=np.uint16)  # bf16 bit patterns


@pytest.mark.parametrize("dtype,layers,h,bs,d,T", [("bf16", 3, 4, 16, 128, 64), ("f16", 1, 2, 32, 64, 9),
                                                   ("f32", 5, 3, 16, 64, 33), ("bf16", 256, 1, 8, 8, 5),
                                                   ("f16", 28, 4, 16, 128, 64)])
def test_write_kv_layers_bit_exact(dtype, layers, h, bs, d, T):
    rng = np.random.default_rng(layers * 7 + T)
    nb = max(8, (T + bs - 1) // bs * 3)
    kcs = [_bits(rng, (nb, h, bs, d), dtype) for _ in range(layers)]
    vcs = [_bits(rng, (nb, h, bs, d), dtype) for _ in range(layers)]
    keys = [_bits(rng, (T, h, d), dtype) for _ in range(layers)]
    vals = [_bits(rng, (T, h, d), dtype) for _ in range(layers)]
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::7] = -1  # padding tokens
    dk = [to_device(x, dtype) for x in kcs]
    dv = [to_device(x, dtype) for x in vcs]
    pa.write_kv_layers([to_device(x, dtype) for x in keys], [to_device(x, dtype) for x in vals], dk, dv,
                       torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert oracle.write_kv_layers(keys, vals, kcs, vcs, slots) == oracle.OK
    for l in range(layers):
        assert np.array_equal(to_host(dk[l], dtype).view(np.uint8), kcs[l].view(np.uint8)), f"key cache {l}"
        assert np.array_equal(to_host(dv[l], dtype).view(np.uint8), vcs[l].view(np.uint8)), f"value cache {l}"
    pa.check_error()


def test_write_kv_layers_flags_a_bad_slot_and_writes_the_rest():
    rng = np.random.default_rng(1)
    kcs = [np.zeros((4, 2, 16, 64), np.float32) for _ in range(2)]
    rows = [rng.standard_normal((3, 2, 64)).astype(np.float32) for _ in range(2)]
    slots = np.array([5, 4 * 16, 17], np.int64)
    dk = [to_device(x, "f32") for x in kcs]
    dv = [to_device(x, "f32") for x in kcs]
    pa.write_kv_layers([to_device(r, "f32") for r in rows], [to_device(-r, "f32") for r in rows], dk, dv,
                       torch.from_numpy(slots).cuda())
    with pytest.raises(pa.PAError) as e:
        pa.check_error()
    assert e.value.status == 6  # PA_ERR_BAD_SLOT
    exp_k = [k.copy() for k in kcs]
    exp_v = [k.copy() for k in kcs]
    assert oracle.write_kv_layers(rows, [-r for r in rows], exp_k, exp_v, slots) == oracle.BAD_SLOT
    for l in range(2):
        assert np.array_equal(to_host(dk[l], "f32"), exp_k[l]) and np.array_equal(to_host(dv[l], "f32"), exp_v[l])


@pytest.mark.parametrize("where", ["device", "pinned"])
def test_apply_table_deltas_bit_exact(where):
    rng = np.random.default_rng(4)
    rows, width = 37, 300
    table = rng.integers(-1, 20000, (rows, width)).astype(np.int32)
    deltas = np.stack([rng.integers(0, rows, 5000), rng.permutation(rows * width)[:5000] % width,
                       rng.integers(0, 20000, 5000)], 1).astype(np.int32)
    # one delta per (row, j): keep the first of duplicates
    _, first = np.unique(deltas[:, 0].astype(np.int64) * width + deltas[:, 1], return_index=True)
    deltas = np.ascontiguousarray(deltas[np.sort(first)])
    dev_table = torch.from_numpy(table).cuda()
    d = torch.from_numpy(deltas)
    d = d.cuda() if where == "device" else d.pin_memory()
    pa.apply_table_deltas(dev_table, d)
    torch.cuda.synchronize()
    exp = table.copy()
    assert oracle.apply_table_deltas(exp, deltas) == oracle.OK
    assert np.array_equal(dev_table.cpu().numpy(), exp)
    pa.check_error()


def test_apply_table_deltas_flags_out_of_range():
    table = torch.zeros(2, 3, dtype=torch.int32, device="cuda")
    deltas = torch.tensor([[0, 0, 7], [1, 2, 9], [2, 0, 1], [0, 3, 5], [-1, 0, 4]], dtype=torch.int32).cuda()
    pa.apply_table_deltas(table, deltas)
    with pytest.raises(pa.PAError) as e:
        pa.check_error()
    assert e.value.status == 5  # PA_ERR_BAD_TABLE
    assert table.cpu().tolist() == [[7, 0, 0], [0, 0, 9]]


def test_delta_maintained_tables_decode_like_full_exports():
    rng = np.random.default_rng(9)
    nb, h, hq, bs, d, rows, width = 400, 2, 8, 16, 128, 8, 48
    pool = pa.BlockPool(nb, bs, free_order=rng.permutation(nb))
    kc = torch.randn(nb, h, bs, d, device="cuda").to(torch.bfloat16)
    vc = torch.randn(nb, h, bs, d, device="cuda").to(torch.bfloat16)
    image = torch.full((rows, width), -1, dtype=torch.int32, device="cuda")
    staging = torch.empty(rows * width, 3, dtype=torch.int32).pin_memory()
    lens_buf = np.empty(rows, np.int32)
    live = [pool.create() for _ in range(rows)]
    for step in range(60):
        for sid in live:
            for _ in range(int(rng.integers(0, 40))):
                if pool.length(sid) >= width * bs:
                    break
                try:
                    pool.append(sid)
                except pa.PoolExhausted:
                    break
        if step % 5 == 4:  # a sequence leaves, a fork of another joins (shared blocks, later copy-on-write)
            pool.release(live.pop(int(rng.integers(len(live)))))
            live.append(pool.fork(live[int(rng.integers(len(live)))]))
        order = [live[i] for i in rng.permutation(len(live))] if step % 3 == 0 else live
        torch.cuda.synchronize()  # the previous step's apply has read the staging
        deltas, lens = pool.table_deltas(order, out=staging.numpy(), lens_out=lens_buf)
        pa.apply_table_deltas(image, staging, len(deltas))
        full, full_lens = pool.block_tables(order, width)
        assert lens.tolist() == full_lens.tolist()
        q = torch.randn(rows, hq, d, device="cuda").to(torch.bfloat16)
        ctx = torch.from_numpy(full_lens).cuda()
        via_deltas = pa.decode(q, kc, vc, image, ctx)
        via_full = pa.decode(q, kc, vc, torch.from_numpy(full).cuda(), ctx)
        torch.cuda.synchronize()
        img = image.cpu().numpy()
        for r, sid in enumerate(order):
            n = (int(full_lens[r]) + bs - 1) // bs
            assert np.array_equal(img[r, :n], full[r, :n])
        assert torch.equal(via_deltas.view(torch.int16), via_full.view(torch.int16))
    pa.check_error()
