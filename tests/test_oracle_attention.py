"""Pins for the oracle's draft/verify attention.

Independent references: torch's scaled_dot_product_attention run in fp64 on
the CPU (a library routine), closed forms (one token, identical keys, one
dominant key), and the identity the verify pass must satisfy: row j equals
decode attention over the full cache extended by new tokens 0..j.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as att
from oracle import kivi


def _bits(x):
    return synth.bf16_bits(np.asarray(x, np.float32))


def _f(b):
    return synth.bf16_to_f32(b).astype(np.float64)


def _sdpa(q, K, V, scale, mask=None):
    """q [n, d], K/V [T, d] fp64 -> [n, d] via torch (library reference)."""
    qt = torch.from_numpy(np.ascontiguousarray(q))[None, None]
    Kt = torch.from_numpy(np.ascontiguousarray(K))[None, None]
    Vt = torch.from_numpy(np.ascontiguousarray(V))[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=m, scale=scale)[0, 0].numpy()


@pytest.mark.parametrize("scale", [1.0, 1 / math.sqrt(64)])
def test_decode_matches_torch_sdpa(scale):
    rng = np.random.default_rng(0)
    B, Hq, Hkv, T, d = 2, 6, 2, 77, 64
    q = _f(_bits(rng.standard_normal((B, Hq, d))))
    K = _f(_bits(rng.standard_normal((B, Hkv, T, d))))
    V = _f(_bits(rng.standard_normal((B, Hkv, T, d))))
    o = att.decode_attention(q, K, V, scale)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            ref = _sdpa(q[b, h][None], K[b, h // G], V[b, h // G], scale)[0]
            assert np.max(np.abs(o[b, h] - ref)) < 1e-12


def test_closed_forms():
    rng = np.random.default_rng(1)
    d = 64
    q = rng.standard_normal((1, 1, d))
    V = rng.standard_normal((1, 1, 10, d))
    # one token: output is that token's value
    assert np.allclose(att.decode_attention(q, rng.standard_normal((1, 1, 1, d)), V[:, :, :1], 1.0)[0, 0], V[0, 0, 0], atol=0)
    # identical keys: uniform weights -> mean of V
    K = np.broadcast_to(rng.standard_normal(d), (1, 1, 10, d))
    assert np.allclose(att.decode_attention(q, K, V, 1.0)[0, 0], V[0, 0].mean(0), atol=1e-14)
    # one key with a logit 50 above the rest: output = its value (to e^-50)
    K = np.zeros((1, 1, 10, d))
    qq = np.zeros((1, 1, d)); qq[0, 0, 0] = 1.0
    K[0, 0, 4, 0] = 50.0
    assert np.allclose(att.decode_attention(qq, K, V, 1.0)[0, 0], V[0, 0, 4], atol=1e-20 + 1e-19 * np.abs(V).max())


def test_round_bf16_matches_rne_of_exact_values():
    # values exactly halfway between bf16 neighbours round to the even one
    one = 1.0
    ulp = 2.0 ** -7
    assert att.round_bf16(np.array([one + ulp / 2]))[0] == one            # tie -> even (1.0)
    assert att.round_bf16(np.array([one + 3 * ulp / 2]))[0] == one + 2 * ulp
    x = np.random.default_rng(3).standard_normal(1000)
    r = att.round_bf16(x)
    # result is on the bf16 grid and within half an ulp
    assert np.array_equal(synth.bf16_to_f32(synth.bf16_bits(r.astype(np.float32))).astype(np.float64), r)
    # within half an ulp: bf16 keeps 8 significant bits, so ulp(x) = 2^(floor(log2|x|) - 7)
    half_ulp = 2.0 ** (np.floor(np.log2(np.abs(x))) - 8)
    assert np.all(np.abs(r - x) <= half_ulp)


def _exact_ramp_kv(B, H, T, d, bits, rng):
    """K/V whose 32-groups are exact ramps, so quantise -> dequantise is exact."""
    q = (1 << bits) - 1
    step = 0.25
    K = np.empty((B, H, T, d), np.float32)
    V = np.empty((B, H, T, d), np.float32)
    for g in range(T // 32):
        base = rng.integers(-8, 8, size=(B, H, 1, d)).astype(np.float32)
        codes = rng.integers(0, q + 1, size=(B, H, 32, d)).astype(np.float32)
        codes[:, :, 0, :] = 0
        codes[:, :, 1, :] = q                                   # min and max present
        K[:, :, 32 * g:32 * g + 32] = base + step * codes
    for t in range(T):
        for cg in range(d // 32):
            base = rng.integers(-8, 8, size=(B, H, 1)).astype(np.float32)
            codes = rng.integers(0, q + 1, size=(B, H, 32)).astype(np.float32)
            codes[..., 0] = 0
            codes[..., 1] = q
            V[:, :, t, 32 * cg:32 * cg + 32] = base + step * codes
    return _bits(K), _bits(V)


@pytest.mark.parametrize("bits", [2, 4])
def test_draft_equals_textbook_when_quantisation_is_exact(bits):
    rng = np.random.default_rng(4)
    B, Hq, Hkv, P, R, d = 2, 4, 2, 64, 5, 64
    Kp, Vp = _exact_ramp_kv(B, Hkv, P, d, bits, rng)
    kc, ksz, vc, vsz = kivi.quant_pack(Kp, Vp, bits)
    tail_k = _bits(rng.standard_normal((B, Hkv, R + 3, d)))
    tail_v = _bits(rng.standard_normal((B, Hkv, R + 3, d)))
    k_cur = _bits(rng.standard_normal((B, Hkv, d)))
    v_cur = _bits(rng.standard_normal((B, Hkv, d)))
    q = _bits(rng.standard_normal((B, Hq, d)) / 8)
    packed_len = np.array([64, 32])
    tail_len = np.array([2, 0])
    step = 3
    o = att.draft_attention(q, kc, ksz, vc, vsz, packed_len, tail_k, tail_v, tail_len, bits, 0.5,
                            k_cur=k_cur, v_cur=v_cur, step=step)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            kvh = h // G
            P_b, R_b = packed_len[b], tail_len[b] + step
            Kall = np.concatenate([_f(Kp[b, kvh, :P_b]), _f(tail_k[b, kvh, :R_b]), _f(k_cur[b, kvh])[None]])
            Vall = np.concatenate([_f(Vp[b, kvh, :P_b]), _f(tail_v[b, kvh, :R_b]), _f(v_cur[b, kvh])[None]])
            ref = _sdpa(_f(q[b, h])[None], Kall, Vall, 0.5)[0]
            assert np.max(np.abs(o[b, h] - ref)) < 1e-12


def test_verify_row_j_is_decode_over_prefix_plus_j_plus_1():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, T, d, k = 2, 4, 1, 50, 64, 3
    q = _bits(rng.standard_normal((B, k + 1, Hq, d)) / 8)
    K = _bits(rng.standard_normal((B, Hkv, T, d)))
    V = _bits(rng.standard_normal((B, Hkv, T, d)))
    kn = _bits(rng.standard_normal((B, k + 1, Hkv, d)))
    vn = _bits(rng.standard_normal((B, k + 1, Hkv, d)))
    plen = np.array([T, 31])
    o = att.verify_attention(q, K, V, kn, vn, plen, 0.7)
    for b in range(B):
        for j in range(k + 1):
            Kj = np.concatenate([_f(K[b, :, :plen[b]]), _f(kn[b, :j + 1]).transpose(1, 0, 2)], axis=1)
            Vj = np.concatenate([_f(V[b, :, :plen[b]]), _f(vn[b, :j + 1]).transpose(1, 0, 2)], axis=1)
            dec = att.decode_attention(_f(q[b, j])[None], Kj[None], Vj[None], 0.7)[0]
            assert np.max(np.abs(o[b, j] - dec)) < 1e-12
    # causality: changing new tokens after j leaves row j unchanged
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[:, 2:], vn2[:, 2:] = _bits(rng.standard_normal(kn2[:, 2:].shape)), _bits(rng.standard_normal(vn2[:, 2:].shape))
    o2 = att.verify_attention(q, K, V, kn2, vn2, plen, 0.7)
    assert np.array_equal(o[:, :2], o2[:, :2]) and not np.allclose(o[:, 2:], o2[:, 2:])
    # torch SDPA with a causal mask over [prefix ; new] for request 0
    b = 0
    Kall = np.concatenate([_f(K[b, 0]), _f(kn[b, :, 0])])
    Vall = np.concatenate([_f(V[b, 0]), _f(vn[b, :, 0])])
    mask = np.zeros((k + 1, T + k + 1), bool)
    for j in range(k + 1):
        mask[j, :T + j + 1] = True
    for h in range(Hq):
        ref = _sdpa(_f(q[b, :, h]), Kall, Vall, 0.7, mask)
        assert np.max(np.abs(o[b, :, h] - ref)) < 1e-12


def test_verify_with_k0_is_decode():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, T, d = 1, 8, 2, 40, 64
    q = _bits(rng.standard_normal((B, 1, Hq, d)))
    K = _bits(rng.standard_normal((B, Hkv, T, d)))
    V = _bits(rng.standard_normal((B, Hkv, T, d)))
    kn = _bits(rng.standard_normal((B, 1, Hkv, d)))
    vn = _bits(rng.standard_normal((B, 1, Hkv, d)))
    o = att.verify_attention(q, K, V, kn, vn, [T], 1.0)
    Kf = np.concatenate([_f(K), _f(kn).transpose(0, 2, 1, 3)], axis=2)
    Vf = np.concatenate([_f(V), _f(vn).transpose(0, 2, 1, 3)], axis=2)
    assert np.max(np.abs(o[:, 0] - att.decode_attention(_f(q[:, 0]), Kf, Vf, 1.0))) < 1e-12
