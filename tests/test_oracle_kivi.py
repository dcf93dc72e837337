"""Pins for the oracle's KIVI-style quantiser and its packed layout.

Nothing here re-derives the oracle's formula: the checks are hand-worked
cases (tests/golden/kivi_cases.json), the nearest-grid-point property, the
error bound s/2, grouping-axis invariants, a hand-written packed word, and
pack/unpack round trips.
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle import kivi

GOLD = os.path.join(os.path.dirname(__file__), "golden", "kivi_cases.json")


def _f32_to_bf16_exact(x):
    x = np.asarray(x, np.float32)
    b = synth.bf16_bits(x)
    assert np.array_equal(synth.bf16_to_f32(b), x), "fixture value not exact in bf16"
    return b


@pytest.mark.parametrize("case", json.load(open(GOLD))["cases"], ids=lambda c: c["name"])
def test_hand_worked_groups(case):
    x = np.asarray(case["x"], np.float32)[None]
    codes, s, z = kivi.quantize_groups(x, case["bits"])
    assert codes[0].tolist() == case["codes"]
    assert s[0] == np.float16(case["scale"])
    assert z[0] == np.float16(case["zero"])


def test_constant_group_dequantises_to_zero_point():
    x = np.full((1, 32), -1.25, np.float32)
    c, s, z = kivi.quantize_groups(x, 4)
    xh = kivi.dequantize(c, np.repeat(s[:, None], 32, 1), np.repeat(z[:, None], 32, 1))
    assert np.all(xh == np.float32(-1.25))


@pytest.mark.parametrize("bits", [2, 4])
def test_nearest_grid_point_and_error_bound(bits):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((400, 32)) * rng.uniform(0.01, 30, (400, 1))).astype(np.float32)
    x = synth.bf16_to_f32(synth.bf16_bits(x))
    codes, s, z = kivi.quantize_groups(x, bits)
    qmax = (1 << bits) - 1
    assert codes.max() <= qmax
    sf = s.astype(np.float64)[:, None]
    zf = z.astype(np.float64)[:, None]
    grid = zf[..., None] + sf[..., None] * np.arange(qmax + 1)            # [n, 1, q+1]
    dist = np.abs(x.astype(np.float64)[..., None] - grid)                  # [n, 32, q+1]
    chosen = np.take_along_axis(dist, codes[..., None].astype(np.int64), -1)[..., 0]
    # the chosen code is a nearest grid point (up to the fp32 rounding of (x-z)/s)
    slack = 4 * np.finfo(np.float32).eps * (np.abs(x) + np.abs(zf) + sf * qmax)
    assert np.all(chosen <= dist.min(-1) + slack)
    # |x - x^| <= s/2 for elements inside [z, z + qmax*s]
    xh = kivi.dequantize(codes, np.repeat(s[:, None], 32, 1), np.repeat(z[:, None], 32, 1)).astype(np.float64)
    inside = (x >= zf) & (x <= zf + qmax * sf)
    err = np.abs(x - xh)
    assert np.all(err[inside] <= (sf / 2 + slack)[np.broadcast_to(True, err.shape) & inside])
    # scale and zero are the fp16 roundings of range/(2^b-1) and of min
    assert np.all(np.abs(s.astype(np.float64) - (x.max(1) - x.min(1)) / qmax) <= 2.0 ** -11 * (x.max(1) - x.min(1)) / qmax + 2.0 ** -25)
    assert np.all(np.abs(z.astype(np.float64) - x.min(1)) <= 2.0 ** -11 * np.abs(x.min(1)) + 2.0 ** -25)


def test_grouping_axes():
    """Keys group along tokens, values along channels."""
    B, H, T, d = 1, 2, 64, 64
    tok = np.arange(T, dtype=np.float32)[:, None] * np.ones((1, d), np.float32)
    ch = np.ones((T, 1), np.float32) * np.arange(d, dtype=np.float32)[None, :]
    # K constant along tokens (value = channel index): every key group is constant
    K = _f32_to_bf16_exact(np.broadcast_to(ch, (B, H, T, d)))
    # V constant along channels (value = token index): every value group is constant
    V = _f32_to_bf16_exact(np.broadcast_to(tok, (B, H, T, d)))
    kc, ks, kz, vc, vs, vz = kivi.quantize_kv(K, V, 2)
    assert np.all(ks == 0) and np.all(vs == 0) and kc.max() == 0 and vc.max() == 0
    assert np.array_equal(kz[0, 0, 0].astype(np.float32), np.arange(d, dtype=np.float32))
    assert np.array_equal(vz[0, 0, :, 0].astype(np.float32), np.arange(T, dtype=np.float32))
    Kh, Vh = kivi.dequantize_kv(kc, ks, kz, vc, vs, vz)
    assert np.array_equal(Kh, synth.bf16_to_f32(K)) and np.array_equal(Vh, synth.bf16_to_f32(V))
    # swapped roles: now every group spans distinct values
    kc2, ks2, *_ = kivi.quantize_kv(V, K, 2)
    assert np.all(ks2 > 0)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_field_tables_are_bijections(bits, d):
    """Every (token, channel) of a group has one field, and the fields of each
    word tile its 32 bits exactly once."""
    for fields in (kivi._k_fields(d, bits), kivi._v_fields(d, bits)):
        assert fields.shape == (32 * d, 4)
        tc = fields[:, 2] * d + fields[:, 3]
        assert np.array_equal(np.sort(tc), np.arange(32 * d))
        cover = np.zeros((d * bits, 32), np.int64)
        for w, p in zip(fields[:, 0], fields[:, 1]):
            for k in range(bits):
                cover[w, (p + k) % 32] += 1
        assert np.all(cover == 1)


def _const_words(pack, code_fn, bits, d):
    t = np.arange(32)[:, None]
    c = np.arange(d)[None, :]
    code = np.broadcast_to(code_fn(t, c), (32, d)).astype(np.uint8)[None, None]
    return pack(code.copy(), bits)


def test_packed_words_by_hand():
    """Words worked out by hand from the field rules.

    b = 2, slot (u, r, e) starts at 16e + 4u + 2(1 - r):
      e = 1 fields: bits 16, 18, ..., 30; a code of 1 in each -> 0x55550000.
      r = 1 fields: 16e + 4u = 0, 4, 8, 12, 16, 20, 24, 28 -> 0x11111111.
    For K, e is the channel's bit 0 and r its bit 1; for V, r is the token's
    bit 0 and e its bit 2.
    b = 4, slot (u, e) starts at 16e + 4u: the e = 1 fields fill bits 16-31,
      so code 15 there -> 0xFFFF0000 and code 1 there -> bits 16, 20, 24, 28 =
      0x11110000."""
    for d in (64, 128):
        assert np.all(_const_words(kivi.pack_kcodes, lambda t, c: c % 2, 2, d) == 0x55550000)
        assert np.all(_const_words(kivi.pack_kcodes, lambda t, c: (c // 2) % 2, 2, d) == 0x11111111)
        assert np.all(_const_words(kivi.pack_vcodes, lambda t, c: t % 2, 2, d) == 0x11111111)
        assert np.all(_const_words(kivi.pack_vcodes, lambda t, c: (t // 4) % 2, 2, d) == 0x55550000)
        assert np.all(_const_words(kivi.pack_kcodes, lambda t, c: 15 * (c % 2), 4, d) == 0xFFFF0000)
        assert np.all(_const_words(kivi.pack_kcodes, lambda t, c: c % 2, 4, d) == 0x11110000)
        assert np.all(_const_words(kivi.pack_vcodes, lambda t, c: (t // 4) % 2, 4, d) == 0x11110000)
        assert np.all(_const_words(kivi.pack_kcodes, lambda t, c: 3 + 0 * c, 2, d) == 0xFFFFFFFF)


def test_single_codes_land_where_the_rules_say():
    """Three codes placed by hand (d = 128 unless noted).

    K, b = 2, token 5, channel 37: a = 1, j = 1; 37 = 32*1 + 4*1 + 2*0 + 1 so
      c = 1, k = 1, r = 0, e = 1; lane 4a + c = 5; fragment j*8 + k = 9 -> word 2,
      u = 1; start 16 + 4 + 2 = 22; stored at (2 // 4)*128 + 4*5 + 2 = 22.
    V, b = 2, token 13, channel 42: 13 = 8*1 + 4*1 + 2*0 + 1 so c = 1, e = 1,
      s = 0, r = 1; 42 = 8*5 + 2 so n = 5, a = 2; lane 9; fragment 0*16 + 5 ->
      word 1, u = 1; start 16 + 4 + 0 = 20; stored at 0 + 36 + 1 = 37.
    K, b = 4, d = 64, token 0, channel 5: a = c = j = 0, k = 1, r = 0, e = 1;
      index 2*(0*4 + 1) + 0 = 2 -> word 0, u = 2; start 16 + 8 = 24:
      code 11 -> 0x0B000000."""
    code = np.zeros((1, 1, 32, 128), np.uint8)
    code[0, 0, 5, 37] = 3
    w = kivi.pack_kcodes(code, 2)[0, 0, 0]
    assert w[22] == 0x00C00000 and np.count_nonzero(w) == 1
    code = np.zeros((1, 1, 32, 128), np.uint8)
    code[0, 0, 13, 42] = 2
    w = kivi.pack_vcodes(code, 2)[0, 0, 0]
    assert w[37] == 0x00200000 and np.count_nonzero(w) == 1
    code = np.zeros((1, 1, 32, 64), np.uint8)
    code[0, 0, 0, 5] = 11
    w = kivi.pack_kcodes(code, 4)[0, 0, 0]
    assert w[0] == 0x0B000000 and np.count_nonzero(w) == 1


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_unpack_bijection(bits):
    rng = np.random.default_rng(11)
    code = rng.integers(0, 1 << bits, size=(2, 3, 96, 128)).astype(np.uint8)
    for pack, unpack in ((kivi.pack_kcodes, kivi.unpack_kcodes), (kivi.pack_vcodes, kivi.unpack_vcodes)):
        words = pack(code, bits)
        assert words.shape == (2, 3, 3, 128 * bits)
        assert np.array_equal(unpack(words, bits, 128), code)
        w = rng.integers(0, 2 ** 32, size=words.shape, dtype=np.uint64).astype(np.uint32)
        assert np.array_equal(pack(unpack(w, bits, 128), bits), w)


def test_meta_layouts():
    """V meta entry p = 8c + 4s + 2r + e holds token 8c + 4e + 2s + r: entry 5
    (c 0, s 1, r 0, e 1) is token 6, entry 19 (c 2, s 0, r 1, e 1) is token 21.
    K meta holds the scales of all channels, then the zeros."""
    rng = np.random.default_rng(5)
    s = rng.standard_normal((2, 2, 64, 4)).astype(np.float16)
    z = rng.standard_normal((2, 2, 64, 4)).astype(np.float16)
    m = kivi.pack_vmeta(s, z)
    assert m.shape == (2, 2, 2, 4, 2, 32)
    assert m[1, 0, 1, 3, 0, 5] == s[1, 0, 32 + 6, 3] and m[1, 0, 1, 3, 1, 5] == z[1, 0, 32 + 6, 3]
    assert m[0, 1, 0, 2, 0, 19] == s[0, 1, 21, 2] and m[0, 1, 0, 2, 1, 19] == z[0, 1, 21, 2]
    s2, z2 = kivi.unpack_vmeta(m)
    assert np.array_equal(s2, s) and np.array_equal(z2, z)
    ks = rng.standard_normal((1, 2, 3, 128)).astype(np.float16)
    kz = rng.standard_normal((1, 2, 3, 128)).astype(np.float16)
    km = kivi.pack_kmeta(ks, kz)
    assert km.shape == (1, 2, 3, 2, 128) and km[0, 1, 2, 0, 77] == ks[0, 1, 2, 77] and km[0, 1, 2, 1, 77] == kz[0, 1, 2, 77]


def test_quant_pack_roundtrip_and_bound_on_workload_inputs():
    w = synth.get("tiny")
    K, V = synth.kv(w)
    kc, ksz, vc, vsz = kivi.quant_pack(K, V, w.bits)
    Kh, Vh = kivi.unpack_dequant(kc, ksz, vc, vsz, w.bits, w.d)
    Kf, Vf = synth.bf16_to_f32(K), synth.bf16_to_f32(V)
    ks = np.repeat(kivi.unpack_kmeta(ksz)[0], 32, axis=2).astype(np.float32)
    vs, _ = kivi.unpack_vmeta(vsz)
    vs = np.repeat(vs, 32, axis=3).astype(np.float32)
    assert np.all(np.abs(Kh - Kf) <= ks / 2 * 1.001 + 1e-3)
    assert np.all(np.abs(Vh - Vf) <= vs / 2 * 1.001 + 1e-3)


def test_eight_bit_words_by_hand():
    """b = 8: slot (u, e) starts at 16e + 8u, two slots per word.
    K codes equal to the channel's bit 0 (e) put a 1 at bits 16 and 24: 0x01010000;
    code 255 in every e = 1 field: 0xFFFF0000.  One code: K, d = 128, token 5,
    channel 37 -> lane 5, j = 1, k = 1, r = 0, e = 1; fragment i = 9, i2 = 2*9 + 0 =
    18 -> word 18 // 2 = 9, u = 0; start 16; stored at (9 // 4)*128 + 4*5 + 9 % 4 = 277:
    code 200 -> 0x00C80000."""
    for d in (64, 128):
        assert np.all(_const_words(kivi.pack_kcodes, lambda t, c: c % 2, 8, d) == 0x01010000)
        assert np.all(_const_words(kivi.pack_kcodes, lambda t, c: 255 * (c % 2), 8, d) == 0xFFFF0000)
        assert np.all(_const_words(kivi.pack_vcodes, lambda t, c: (t // 4) % 2, 8, d) == 0x01010000)
    code = np.zeros((1, 1, 32, 128), np.uint8)
    code[0, 0, 5, 37] = 200
    w = kivi.pack_kcodes(code, 8)[0, 0, 0]
    assert w.shape == (1024,) and w[277] == 0x00C80000 and np.count_nonzero(w) == 1
