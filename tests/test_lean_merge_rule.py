"""The lean schedule's merge assignment rule, checked exhaustively on the host.

The lean decode lays the pages of all (sequence, kv head, head chunk) units end to end and cuts
them into equal shares of q pages, one per consumer warp; a unit is cut only where a share ends.
When units outnumber warps the merge kernel runs one CTA per boundary w (the first page of warp
w, P = w * q): the CTA takes the unit holding page P and merges it only if P lies strictly
inside it and no earlier boundary does (w == first // q + 1).  This test restates that rule and
checks that every unit cut by a boundary is merged exactly once and no whole unit is touched,
for many random length mixes (the GPU tests run the kernel itself).
"""
import numpy as np
import pytest


def units_and_share(lens, upb, block_size, warps):
    pages = [(int(L) + block_size - 1) // block_size for L in lens]
    units = []  # (first, nb) in the global page order: sequence-major, then unit
    pre = 0
    for n in pages:
        for uu in range(upb):
            units.append((pre * upb + uu * n, n))
        pre += n
    total = pre * upb
    q = (total + warps - 1) // warps
    return units, q


def boundary_assignment(lens, upb, block_size, warps):
    units, q = units_and_share(lens, upb, block_size, warps)
    merged = []
    for w in range(1, max(warps - 1, 1) + 1):
        P = w * q
        hit = [(f, n) for f, n in units if n > 0 and f <= P < f + n]
        if not hit:
            continue
        first, n = hit[0]
        if first == P or first // q + 1 != w:
            continue
        merged.append(first)
    return units, q, merged


@pytest.mark.parametrize("seed", range(40))
def test_each_cut_unit_is_merged_once(seed):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 300))
    upb = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32]))
    warps = int(rng.integers(2, 400))
    lens = rng.integers(0, 900, b)
    lens[rng.random(b) < 0.2] = 0  # empty contexts
    units, q, merged = boundary_assignment(lens, upb, bs, warps)
    if q == 0:
        assert merged == []
        return
    cut = sorted(f for f, n in units if n > 0 and f // q != (f + n - 1) // q)
    assert sorted(merged) == cut
    assert len(merged) == len(set(merged))


def test_boundaries_on_unit_starts_merge_nothing():
    # every unit exactly one share long: boundaries fall on unit starts, nothing is cut
    lens = [16 * 4] * 10
    units, q, merged = boundary_assignment(lens, 1, 16, warps=10)
    assert q == 4 and merged == []
