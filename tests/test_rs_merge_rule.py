"""The row-split schedule's record rule, checked on the host for many length mixes.

The row-split decode (multi-query, 9..32 query rows per kv head) lays the pages of all
(sequence, kv head) units end to end, sequence-major, and cuts them into equal shares of
S = ceil(total / CTAs) pages, one per CTA.  A CTA walks its share unit by unit: a unit that lies
wholly inside the share is written out directly; a cut one leaves a record in slot 0 when it is
the share's first unit and in slot 1 otherwise.  The merge recomputes, per unit, the first CTA
c0 = start // S and the count n of CTAs its pages span, and reads slot 1 of c0 (slot 0 when the
unit starts the share) and slot 0 of every later CTA.  This test restates both sides and checks
that every record written is read exactly once, by the unit that wrote it, and that exactly the
units the merge skips (n == 1) were written out directly (the GPU tests run the kernels).
"""
import bisect

import numpy as np
import pytest


def layout(lens, hkv, block_size):
    nblk = [(int(L) + block_size - 1) // block_size for L in lens]
    pre = [0]
    for n in nblk:
        pre.append(pre[-1] + n)
    return nblk, pre


def locate(pre, hkv, g):
    # the last sequence whose first page is at or before g (sequences without pages are skipped)
    b = bisect.bisect_right([p * hkv for p in pre[:-1]], g) - 1
    nb = pre[b + 1] - pre[b]
    r = g - pre[b] * hkv
    return b, r // nb, r % nb, nb


def decode_side(lens, hkv, block_size, ctas):
    nblk, pre = layout(lens, hkv, block_size)
    total = pre[-1] * hkv
    share = -(-total // ctas)
    records, direct = {}, set()
    for c in range(ctas):
        g0 = min(total, c * share)
        g1 = min(total, g0 + share)
        g = g0
        while g < g1:
            b, kvh, j, nb = locate(pre, hkv, g)
            cnt = min(g1 - g, nb - j)
            if cnt == nb:
                direct.add((b, kvh))
            else:
                key = (c, 0 if g == g0 else 1)
                assert key not in records, "two cut units in one record slot"
                records[key] = (b, kvh)
            g += cnt
    return records, direct, share


def merge_side(lens, hkv, block_size, ctas):
    nblk, pre = layout(lens, hkv, block_size)
    total = pre[-1] * hkv
    reads, skipped, zeros = {}, set(), set()
    for b, nb in enumerate(nblk):
        for kvh in range(hkv):
            if nb == 0:
                zeros.add((b, kvh))
                continue
            share = -(-total // ctas)
            start = pre[b] * hkv + kvh * nb
            c0 = start // share
            n = (start + nb - 1) // share - c0 + 1
            assert c0 + n - 1 < ctas
            if n <= 1:
                skipped.add((b, kvh))
                continue
            slot0 = 0 if start == c0 * share else 1
            for p in range(n):
                key = (c0 + p, slot0 if p == 0 else 0)
                assert key not in reads, "a record read by two units"
                reads[key] = (b, kvh)
    return reads, skipped, zeros


def check(lens, hkv, block_size, ctas):
    records, direct, _ = decode_side(lens, hkv, block_size, ctas)
    reads, skipped, zeros = merge_side(lens, hkv, block_size, ctas)
    assert records == reads
    assert direct == skipped
    units = {(b, k) for b in range(len(lens)) for k in range(hkv)}
    assert direct | set(records.values()) | zeros == units


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 152, 456])
@pytest.mark.parametrize("hkv", [1, 2, 4, 8])
def test_random_length_mixes(ctas, hkv):
    rng = np.random.default_rng(ctas * 10 + hkv)
    for _ in range(40):
        B = int(rng.integers(1, 70))
        lens = rng.integers(0, 3000, size=B)
        lens[rng.random(B) < 0.2] = 0  # empty contexts
        check(lens, hkv, 16, ctas)


def test_edge_mixes():
    check([0, 0, 0], 4, 16, 456)             # nothing to stream: every row zeroed by the merge
    check([1], 1, 16, 456)                   # one page against many CTAs
    check([4096], 1, 16, 456)                # one unit over 256 single-page shares
    check([16, 16, 16, 16], 2, 16, 8)        # shares equal to units: no cut
    check([17, 0, 33, 5000, 3], 4, 32, 152)  # block size 32


def test_verify_workload_shape():
    rng = np.random.default_rng(0)
    check(rng.integers(512, 4097, size=64), 4, 16, 456)
