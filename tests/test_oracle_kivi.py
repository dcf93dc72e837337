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


def test_packed_word_by_hand():
    """d=32, b=4: token t, channel c has code c % 16.  Word w of a token holds
    channels 8w..8w+7, code j at bits 4j..4j+3: w=0 -> 0x76543210, w=1 ->
    0xFEDCBA98, w=2 -> 0x76543210, w=3 -> 0xFEDCBA98."""
    code = np.broadcast_to((np.arange(32) % 16).astype(np.uint8), (1, 1, 64, 32)).copy()
    words = kivi.pack_codes(code, 4)
    assert words.shape == (1, 1, 2, 4, 32)
    assert np.all(words[0, 0, :, 0, :] == 0x76543210)
    assert np.all(words[0, 0, :, 1, :] == 0xFEDCBA98)
    assert np.all(words[0, 0, :, 2, :] == 0x76543210)
    # b=2: channel c code c % 4 -> 16 codes per word: 0b11100100 repeated = 0xE4E4E4E4
    code2 = np.broadcast_to((np.arange(32) % 4).astype(np.uint8), (1, 1, 32, 32)).copy()
    assert np.all(kivi.pack_codes(code2, 2) == 0xE4E4E4E4)
    # the word index runs over tokens fastest: token t lands in lane t
    code3 = np.zeros((1, 1, 32, 32), np.uint8)
    code3[0, 0, 5, 9] = 3                                  # token 5, channel 9 (word 1 at b=4, j=1)
    w3 = kivi.pack_codes(code3, 4)
    assert w3[0, 0, 0, 1, 5] == 3 << 4 and np.count_nonzero(w3) == 1


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_unpack_bijection(bits):
    rng = np.random.default_rng(11)
    code = rng.integers(0, 1 << bits, size=(2, 3, 96, 128)).astype(np.uint8)
    words = kivi.pack_codes(code, bits)
    assert np.array_equal(kivi.unpack_codes(words, bits, 128), code)
    # and every word is reachable: unpack then pack
    w = rng.integers(0, 2 ** 32, size=words.shape, dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(kivi.pack_codes(kivi.unpack_codes(w, bits, 128), bits), w)


def test_vmeta_layout_roundtrip():
    rng = np.random.default_rng(5)
    s = rng.standard_normal((2, 2, 64, 4)).astype(np.float16)
    z = rng.standard_normal((2, 2, 64, 4)).astype(np.float16)
    m = kivi.pack_vmeta(s, z)
    assert m.shape == (2, 2, 2, 4, 32, 2)
    # (g, cg, t) holds token 32g+t of channel group cg
    assert m[1, 0, 1, 3, 7, 0] == s[1, 0, 32 + 7, 3] and m[1, 0, 1, 3, 7, 1] == z[1, 0, 39, 3]
    s2, z2 = kivi.unpack_vmeta(m)
    assert np.array_equal(s2, s) and np.array_equal(z2, z)


def test_quant_pack_roundtrip_and_bound_on_workload_inputs():
    w = synth.get("tiny")
    K, V = synth.kv(w)
    kc, ksz, vc, vsz = kivi.quant_pack(K, V, w.bits)
    Kh, Vh = kivi.unpack_dequant(kc, ksz, vc, vsz, w.bits, w.d)
    Kf, Vf = synth.bf16_to_f32(K), synth.bf16_to_f32(V)
    ks = np.repeat(ksz[..., 0], 32, axis=2).astype(np.float32)
    vs, _ = kivi.unpack_vmeta(vsz)
    vs = np.repeat(vs, 32, axis=3).astype(np.float32)
    assert np.all(np.abs(Kh - Kf) <= ks / 2 * 1.001 + 1e-3)
    assert np.all(np.abs(Vh - Vf) <= vs / 2 * 1.001 + 1e-3)
