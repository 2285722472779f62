"""Pins for the FP8 (E4M3) KV-cache oracle.

* decoding: every one of the 256 codes against torch's float8_e4m3fn cast (a library
  routine), plus closed-form values (1, 448, the smallest subnormal and normal, NaN);
* encoding: random values and every midpoint between neighbouring codes against
  torch's cast (round to nearest, ties to the even mantissa); saturation to 448 and NaN
  by their definition; the half-step error bound on a dense sweep;
* the FP8 write: the stored codes are the encoding of float32(x) / float32(scale) at the
  slot (numpy division + torch cast, an independent route), every other byte unchanged;
* the FP8 decode: equal to dense softmax attention on the dequantised, gathered K/V
  (numpy), and to the unscaled oracle on an f32 cache holding the same values when the
  scales are powers of two (the products are then exact in float32).
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle


def torch_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def torch_encode(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_codes_matches_library_cast():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.element_to_double(codes, "e4m3")
    ref = torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x07] == 7 * 2.0 ** -9
    assert got[0x80] == 0.0 and np.signbit(got[0x80])


def test_encode_matches_library_cast_on_random_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(50000) * 1e-2,
                        rng.uniform(-447.9, 447.9, 20000)]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), torch_encode(x))


def test_encode_midpoints_round_to_even():
    pos = oracle.element_to_double(np.arange(0x7F, dtype=np.uint8), "e4m3")  # 0 .. 448, increasing
    assert np.all(np.diff(pos) > 0)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # exact in float32
    got = oracle.e4m3_encode(mids)
    lower = np.arange(0x7E, dtype=np.uint8)
    expect = np.where(lower % 2 == 0, lower, lower + 1)  # the even code of the two neighbours
    assert np.array_equal(got, expect)
    assert np.array_equal(got, torch_encode(mids))
    assert np.array_equal(oracle.e4m3_encode(-mids), expect | 0x80)


def test_encode_saturates_and_keeps_nan():
    x = np.array([448, 449, 463.9, 464, 480, 1e30, np.inf, -500, -np.inf, np.nan, -0.0, 0.0], np.float32)
    got = oracle.e4m3_encode(x)
    assert got[:6].tolist() == [0x7E] * 6 and got[6] == 0x7E
    assert got[7] == 0xFE and got[8] == 0xFE
    assert got[9] & 0x7F == 0x7F
    assert got[10] == 0x80 and got[11] == 0x00


def test_encode_error_is_within_half_a_step():
    x = np.linspace(-447, 447, 400001, dtype=np.float32)
    back = oracle.element_to_double(oracle.e4m3_encode(x[::97]), "e4m3")
    xs = x[::97].astype(np.float64)
    step = np.where(np.abs(xs) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(xs), 1e-30))) - 3))
    assert np.all(np.abs(back - xs) <= step / 2)


def _fp8_case(seed, num_seqs=3, hkv=2, hq=6, bs=16, d=64, lens=(1, 17, 40), pow2_scales=False, q_dtype="bf16"):
    rng = np.random.default_rng(seed)
    nb = 12
    kc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    vc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x11  # no NaN codes in a written cache
    vc[(vc & 0x7F) == 0x7F] = 0x22
    if pow2_scales:
        ks = (2.0 ** rng.integers(-8, -3, (nb, hkv))).astype(np.float32)
        vs = (2.0 ** rng.integers(-8, -3, (nb, hkv))).astype(np.float32)
    else:
        ks = rng.uniform(0.002, 0.02, (nb, hkv)).astype(np.float32)
        vs = rng.uniform(0.002, 0.02, (nb, hkv)).astype(np.float32)
    perm = rng.permutation(nb)
    width = 3
    bt = np.full((num_seqs, width), -1, np.int32)
    k = 0
    for b, L in enumerate(lens):
        n = (L + bs - 1) // bs
        bt[b, :n] = perm[k:k + n]
        k += n
    qf = rng.standard_normal((num_seqs, hq, d)).astype(np.float32)
    q = (torch.from_numpy(qf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) if q_dtype == "bf16"
         else qf)
    return q, kc, vc, ks, vs, bt, np.array(lens, np.int32), 1 / np.sqrt(d)


def test_decode_fp8_equals_dense_attention_on_dequantised_kv():
    q, kc, vc, ks, vs, bt, lens, scale = _fp8_case(1)
    got = oracle.decode_fp8(q, "bf16", kc, vc, ks, vs, bt, lens, scale)
    qd = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).double().numpy()
    hkv, bs = kc.shape[1], kc.shape[2]
    g = q.shape[1] // hkv
    for b, L in enumerate(lens):
        blocks = bt[b, :(L + bs - 1) // bs]
        for qh in range(q.shape[1]):
            h = qh // g
            K = (torch_decode(kc[blocks, h]) * ks[blocks, h][:, None, None].astype(np.float64)).reshape(-1, 64)[:L]
            V = (torch_decode(vc[blocks, h]) * vs[blocks, h][:, None, None].astype(np.float64)).reshape(-1, 64)[:L]
            ref = softmax(scale * K @ qd[b, qh]) @ V
            np.testing.assert_allclose(got[b, qh], ref, rtol=1e-12, atol=1e-12)


def test_decode_fp8_equals_unscaled_oracle_with_power_of_two_scales():
    q, kc, vc, ks, vs, bt, lens, scale = _fp8_case(2, pow2_scales=True, q_dtype="f32")
    got = oracle.decode_fp8(q, "f32", kc, vc, ks, vs, bt, lens, scale)
    kf = (torch_decode(kc) * ks[:, :, None, None]).astype(np.float32)
    vf = (torch_decode(vc) * vs[:, :, None, None]).astype(np.float32)
    assert np.array_equal(kf.astype(np.float64), torch_decode(kc) * ks[:, :, None, None])  # exact
    ref = oracle.decode(q, kf, vf, bt, lens, "f32", scale)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_decode_fp8_scale_is_per_block_and_head():
    # doubling one (block, head) scale of V doubles exactly that block's contribution
    q, kc, vc, ks, vs, bt, lens, scale = _fp8_case(3, lens=(40, 1, 17))
    base = oracle.decode_fp8(q, "bf16", kc, vc, ks, vs, bt, lens, scale)
    vs2 = vs.copy()
    vs2[bt[1, 0], 0] *= 2  # sequence 1 (L = 1) reads only block bt[1, 0]; kv head 0 serves heads 0..2
    got = oracle.decode_fp8(q, "bf16", kc, vc, ks, vs2, bt, lens, scale)
    np.testing.assert_allclose(got[1, :3], 2 * base[1, :3], rtol=1e-14)
    np.testing.assert_array_equal(got[1, 3:], base[1, 3:])
    np.testing.assert_array_equal(got[0], base[0]) if bt[1, 0] not in bt[0] else None


@pytest.mark.parametrize("src", ["bf16", "f32", "f16"])
def test_write_fp8_stores_the_encoding_of_x_over_scale(src):
    rng = np.random.default_rng(4)
    nb, hkv, bs, d, T = 5, 2, 4, 16, 9
    kc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    vc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    k0, v0 = kc.copy(), vc.copy()
    ks = rng.uniform(0.01, 0.1, (nb, hkv)).astype(np.float32)
    vs = rng.uniform(0.01, 0.1, (nb, hkv)).astype(np.float32)
    xf = (rng.standard_normal((2, T, hkv, d)) * 8).astype(np.float32)
    xf[0, 0, 0, :3] = [1e4, -1e4, np.nan]  # saturating and NaN inputs
    if src == "bf16":
        key = torch.from_numpy(xf[0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        val = torch.from_numpy(xf[1]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        kx = torch.from_numpy(key.view(np.int16)).view(torch.bfloat16).float().numpy()
        vx = torch.from_numpy(val.view(np.int16)).view(torch.bfloat16).float().numpy()
    elif src == "f16":
        key, val = xf[0].astype(np.float16), xf[1].astype(np.float16)
        kx, vx = key.astype(np.float32), val.astype(np.float32)
    else:
        key, val, kx, vx = xf[0], xf[1], xf[0], xf[1]
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int64)
    slots[4] = -1
    assert oracle.write_kv_fp8(key, val, src, kc, vc, ks, vs, slots) == oracle.OK
    written = set()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), bs)
        written.add((blk, off))
        for h in range(hkv):
            # torch's cast maps magnitudes past the largest code to NaN: the saturation is the definition's
            qk, qv = np.float32(kx[t, h]) / ks[blk, h], np.float32(vx[t, h]) / vs[blk, h]
            ek = np.where(np.abs(qk) >= 448, np.where(qk < 0, 0xFE, 0x7E), torch_encode(qk))
            ev = np.where(np.abs(qv) >= 448, np.where(qv < 0, 0xFE, 0x7E), torch_encode(qv))
            nan = np.isnan(kx[t, h])
            np.testing.assert_array_equal(kc[blk, h, off][~nan], ek[~nan])
            assert np.all(kc[blk, h, off][nan] & 0x7F == 0x7F)
            np.testing.assert_array_equal(vc[blk, h, off], ev)
    for blk in range(nb):
        for off in range(bs):
            if (blk, off) not in written:
                np.testing.assert_array_equal(kc[blk, :, off], k0[blk, :, off])
                np.testing.assert_array_equal(vc[blk, :, off], v0[blk, :, off])
    assert oracle.write_kv_fp8(key[:1], val[:1], src, kc, vc, ks, vs, np.array([nb * bs], np.int64)) == oracle.BAD_SLOT
