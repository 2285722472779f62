"""Pins for the multi-layer write oracle, the table-delta oracle and the allocator
model's delta export.

* multi-layer write: layer l's cache holds layer l's rows at the shared slots,
  read through numpy's own slot-major view (a transpose/reshape), and nothing
  else changes; rows tagged with their layer catch a layer mix-up;
* delta application: a hand-checked case, out-of-range entries skipped and reported;
* delta export: after random pool operations and random row assignments, a
  persistent table image patched only with the exported deltas agrees with the
  full export on every entry the decode reads; a sequence re-exported to its own
  row names only entries that changed; a sequence in a new row names all of them.
"""
import numpy as np
import pytest

import oracle
from oracle.block_pool import SequencePool


def slot_major(cache):
    nb, h, bs, d = cache.shape
    return cache.transpose(1, 0, 2, 3).reshape(h, nb * bs, d)


def test_write_kv_layers_writes_each_layer_its_own_rows():
    rng = np.random.default_rng(2)
    layers, nb, h, bs, d, T = 3, 5, 2, 4, 8, 7
    kcs = [rng.standard_normal((nb, h, bs, d)).astype(np.float32) for _ in range(layers)]
    vcs = [rng.standard_normal((nb, h, bs, d)).astype(np.float32) for _ in range(layers)]
    before = [(k.copy(), v.copy()) for k, v in zip(kcs, vcs)]
    keys = [(np.full((T, h, d), 100.0 * (l + 1)) + np.arange(T)[:, None, None]).astype(np.float32)
            for l in range(layers)]
    vals = [-k for k in keys]
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[3] = -1
    assert oracle.write_kv_layers(keys, vals, kcs, vcs, slots) == oracle.OK
    for l in range(layers):
        ks, vs = slot_major(kcs[l]), slot_major(vcs[l])
        ks0, vs0 = slot_major(before[l][0]), slot_major(before[l][1])
        written = [int(s) for s in slots if s >= 0]
        for t, s in enumerate(slots):
            if s >= 0:
                np.testing.assert_array_equal(ks[:, s], keys[l][t])
                np.testing.assert_array_equal(vs[:, s], vals[l][t])
        rest = [s for s in range(nb * bs) if s not in written]
        np.testing.assert_array_equal(ks[:, rest], ks0[:, rest])
        np.testing.assert_array_equal(vs[:, rest], vs0[:, rest])


def test_write_kv_layers_reports_a_bad_slot():
    kc = [np.zeros((2, 1, 2, 4), np.float32) for _ in range(2)]
    vc = [np.zeros_like(k) for k in kc]
    rows = [np.ones((1, 1, 4), np.float32)] * 2
    assert oracle.write_kv_layers(rows, rows, kc, vc, np.array([4], np.int64)) == oracle.BAD_SLOT


def test_apply_table_deltas_hand_case():
    t = np.full((2, 3), -1, np.int32)
    st = oracle.apply_table_deltas(t, np.array([[0, 0, 7], [1, 2, 9], [0, 1, 4], [2, 0, 1], [0, 3, 5]]))
    assert st == oracle.BAD_TABLE
    assert t.tolist() == [[7, 4, -1], [-1, -1, 9]]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_delta_export_keeps_a_device_image_current(seed):
    rng = np.random.default_rng(seed)
    bs, nb, width, rows = 4, 200, 64, 12
    pool = SequencePool(nb, bs, free_order=rng.permutation(nb))
    image = np.full((rows, width), -1, np.int32)  # the device-resident tables
    holder = {}  # row -> sequence whose entries the image row holds
    live = []
    for step in range(400):
        op = rng.integers(0, 8)
        if op == 0 or not live:
            live.append(pool.create())
        elif op == 1 and len(live) < 40:
            live.append(pool.fork(live[rng.integers(len(live))]))
        elif op == 2:
            pool.release(live.pop(rng.integers(len(live))))
        else:
            for sid in rng.choice(live, size=min(len(live), 5), replace=False):
                try:
                    pool.append(int(sid))
                except MemoryError:
                    pass
        if step % 3 == 0 and live:
            batch = [int(x) for x in rng.permutation(live)[:rows]]
            # rows whose image still holds this sequence from its last export
            kept = {r for r, sid in enumerate(batch) if holder.get(r) == sid}
            deltas, lens = pool.table_deltas(batch)
            for r, j, b in deltas:
                if r in kept:
                    assert image[r, j] != b, "an unchanged entry was exported again"
            new_rows = set(range(len(batch))) - kept
            for r in new_rows:
                assert sorted(j for rr, j, _ in deltas if rr == r) == list(range(len(pool.tables[batch[r]])))
            assert oracle.apply_table_deltas(image, np.array(deltas, np.int64).reshape(-1, 3)) == oracle.OK
            full, full_lens = pool.block_tables(batch, width)
            assert lens == full_lens.tolist()
            for r, sid in enumerate(batch):
                n = len(pool.tables[sid])
                np.testing.assert_array_equal(image[r, :n], full[r, :n])
                holder[r] = sid
