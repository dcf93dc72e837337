"""vc_quant_kv on the GPU vs the oracle.

Bit-exact: packed code words, fp16 scale/zero (compared as values, so -0 == +0),
dequantised values, append/commit state, selected indices (with the near-tie
rule below), gathered rows.  Token scores: fp32 GPU vs fp64 oracle.
"""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import kivi, tokendrop, loop as oloop

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    from verify_compressed_kv_gb300 import _lib
    return _lib


def alloc_packed(vc, s, T_cap):
    from gpu_util import DEV
    kcb, kszb, vcb, vszb = vc.vc_quant_packed_bytes(s, T_cap)
    return (torch.zeros(kcb // 4, dtype=torch.int32, device=DEV), torch.zeros(kszb // 2, dtype=torch.int16, device=DEV),
            torch.zeros(vcb // 4, dtype=torch.int32, device=DEV), torch.zeros(vszb // 2, dtype=torch.int16, device=DEV))


def gpu_pack(vc, K, V, bits, T_cap=None):
    from gpu_util import dev
    B, H, T, d = K.shape
    T_cap = T if T_cap is None else T_cap
    s = vc.shape(B, H, H, d, bits=bits)
    kc, ksz, vcc, vsz = alloc_packed(vc, s, T_cap)
    vc.vc_quant_kv_pack(s, T, T_cap, dev(K), dev(V), kc, ksz, vcc, vsz)
    torch.cuda.synchronize()
    return s, (kc, ksz, vcc, vsz)


def to_np(packed, B, H, T_cap, d, bits):
    kc, ksz, vcc, vsz = packed
    NG = T_cap // 32
    return (kc.cpu().numpy().view(np.uint32).reshape(B, H, NG, d * bits),
            ksz.cpu().numpy().view(np.float16).reshape(B, H, NG, 2, d),
            vcc.cpu().numpy().view(np.uint32).reshape(B, H, NG, d * bits),
            vsz.cpu().numpy().view(np.float16).reshape(B, H, NG, d // 32, 2, 32))


def assert_packed_equal(got, want, NG=None):
    names = ["kc", "ksz", "vc", "vsz"]
    for n, g, w in zip(names, got, want):
        if NG is not None:
            g = g[:, :, :NG]
            w = w[:, :, :NG]
        if g.dtype == np.float16:
            assert np.array_equal(g.astype(np.float32), w.astype(np.float32)), f"{n} differs"
        else:
            assert np.array_equal(g, w), f"{n} differs at {np.argwhere(g != w)[:5]}"


@pytest.mark.parametrize("B,H,T,d,bits", [(1, 1, 512, 64, 4), (2, 2, 1024, 128, 2), (2, 3, 96, 128, 4),
                                          (1, 2, 64, 64, 2), (2, 2, 256, 128, 8), (1, 1, 96, 64, 8)])
def test_pack_bit_exact(vc, B, H, T, d, bits):
    w = synth.get("mistral", B=B, Hkv=H, Hq=H, T=T, d=d, bits=bits)
    K, V = synth.kv(w)
    _, packed = gpu_pack(vc, K, V, bits, T_cap=T + 64)
    got = to_np(packed, B, H, T + 64, d, bits)
    want = kivi.quant_pack(K, V, bits)
    assert_packed_equal(got, want, NG=T // 32)


def tie_grid(rng, shape, bits, step, group_axis):
    """bf16 bits of values on a grid of half a scale step, with every 32-group's min
    and max pinned to 0 and qmax*step: (x - z)/s is an exact half-integer for half
    of the elements, so round-half-even decides their codes."""
    qmax = (1 << bits) - 1
    m = rng.integers(0, min(2 * qmax, 256) + 1, size=shape)          # <= 8 significant bits
    x = m.astype(np.float32) * np.float32(step / 2)
    x = np.moveaxis(x, group_axis, -1).copy()
    grp = x.reshape(*x.shape[:-1], -1, 32)
    grp[..., 0] = 0.0
    grp[..., 1] = qmax * step
    x = np.moveaxis(grp.reshape(x.shape), -1, group_axis)
    b = x.astype(np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "grid values must be exact in bf16"
    return np.ascontiguousarray((b >> 16).astype(np.uint16))


@pytest.mark.parametrize("bits,step", [(2, 0.5), (2, 1.5), (4, 0.125), (4, 0.375), (8, 0.0625)])
def test_pack_bit_exact_at_exact_ties(vc, bits, step):
    """Quotients that are exact half-integers (and their neighbours on the grid)
    must round half to even exactly as the oracle's fp32 division does."""
    B, H, T, d = 2, 2, 256, 128
    rng = np.random.default_rng(bits * 100 + int(step * 64))
    K = tie_grid(rng, (B, H, T, d), bits, step, group_axis=2)     # keys: groups along tokens
    V = tie_grid(rng, (B, H, T, d), bits, step, group_axis=3)     # values: groups along channels
    _, packed = gpu_pack(vc, K, V, bits)
    got = to_np(packed, B, H, T, d, bits)
    want = kivi.quant_pack(K, V, bits)
    assert_packed_equal(got, want)


def wide_range(rng, shape, group_axis):
    """bf16 bits of groups with magnitudes 2^-24 .. 2^10 and offsets of a few
    magnitudes: scales from fp16 subnormals (and zero) to large, every exponent of
    the quotient path."""
    x = rng.standard_normal(shape).astype(np.float32)
    x = np.moveaxis(x, group_axis, -1)
    g = x.reshape(*x.shape[:-1], -1, 32)
    mag = np.exp2(rng.uniform(-24, 10, size=g.shape[:-1] + (1,))).astype(np.float32)
    off = (rng.standard_normal(g.shape[:-1] + (1,)) * 4).astype(np.float32) * mag
    x = np.moveaxis((g * mag + off).reshape(x.shape), -1, group_axis)
    b = np.ascontiguousarray(x).view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)        # RNE to bf16


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_pack_bit_exact_wide_value_range(vc, bits):
    B, H, T, d = 1, 4, 2048, 128
    rng = np.random.default_rng(40 + bits)
    K = wide_range(rng, (B, H, T, d), 2)
    V = wide_range(rng, (B, H, T, d), 3)
    _, packed = gpu_pack(vc, K, V, bits)
    assert_packed_equal(to_np(packed, B, H, T, d, bits), kivi.quant_pack(K, V, bits))


def test_pack_hand_worked_groups(vc):
    """The golden groups, placed as key channels and as value channel groups."""
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "kivi_cases.json")))["cases"]
    for c in cases:
        x = np.asarray(c["x"], np.float32)
        d = 64
        K = np.zeros((1, 1, 32, d), np.float32)
        V = np.zeros((1, 1, 32, d), np.float32)
        K[0, 0, :, 5] = x                    # key channel 5 across the 32 tokens
        V[0, 0, 7, 32:] = x                  # value token 7, channel group 1
        Kb, Vb = synth.bf16_bits(K), synth.bf16_bits(V)
        _, packed = gpu_pack(vc, Kb, Vb, c["bits"])
        kc, ksz, vcc, vsz = to_np(packed, 1, 1, 32, d, c["bits"])
        kcode = kivi.unpack_kcodes(kc, c["bits"], d)
        vcode = kivi.unpack_vcodes(vcc, c["bits"], d)
        assert kcode[0, 0, :, 5].tolist() == c["codes"], c["name"]
        assert vcode[0, 0, 7, 32:].tolist() == c["codes"], c["name"]
        ks, kz = kivi.unpack_kmeta(ksz)
        vs, vz = kivi.unpack_vmeta(vsz)
        assert ks[0, 0, 0, 5] == np.float16(c["scale"]) and kz[0, 0, 0, 5] == np.float16(c["zero"])
        assert vs[0, 0, 7, 1] == np.float16(c["scale"]) and vz[0, 0, 7, 1] == np.float16(c["zero"])


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_unpack_bit_exact(vc, bits):
    from gpu_util import DEV
    w = synth.get("mistral", B=2, Hkv=2, Hq=2, T=256, bits=bits)
    K, V = synth.kv(w)
    s, packed = gpu_pack(vc, K, V, bits)
    Kh = torch.empty((2, 2, 256, 128), dtype=torch.float32, device=DEV)
    Vh = torch.empty_like(Kh)
    vc.vc_quant_kv_unpack(s, 256, 256, *packed, Kh, Vh)
    oK, oV = kivi.unpack_dequant(*kivi.quant_pack(K, V, bits), bits, 128)
    assert np.array_equal(Kh.cpu().numpy(), oK) and np.array_equal(Vh.cpu().numpy(), oV)


def test_pack_full_size_sampled(vc):
    """Mistral-shaped layer at full size: every slice packed on the GPU in one
    launch; sampled (request, head) slices checked bit for bit."""
    w = synth.get("mistral")
    K, V = synth.kv(w)
    _, packed = gpu_pack(vc, K, V, w.bits)
    got = to_np(packed, w.B, w.Hkv, w.T, w.d, w.bits)
    for (b, h) in [(0, 0), (3, 5), (w.B - 1, w.Hkv - 1)]:
        want = kivi.quant_pack(K[b:b + 1, h:h + 1], V[b:b + 1, h:h + 1], w.bits)
        assert_packed_equal([g[b:b + 1, h:h + 1] for g in got], want)


@pytest.mark.parametrize("bits,k", [(4, 4), (2, 16), (2, 33), (8, 7)])
def test_append_matches_oracle_commit(vc, bits, k):
    from gpu_util import dev, DEV
    B, H, d = 3, 2, 64 if bits == 4 else 128
    rng = np.random.default_rng(k)
    T0 = [64, 96, 32]
    T_cap = 512
    tail_cap = 32 + k + 1
    # initial draft caches: packed prefixes of different lengths, empty tails
    w = synth.get("mistral", B=B, Hkv=H, Hq=H, T=max(T0), d=d, bits=bits)
    K, V = synth.kv(w)
    s = vc.shape(B, H, H, d, k=k, bits=bits)
    packed = alloc_packed(vc, s, T_cap)
    # pack each request's prefix (pack writes groups 0..T/32-1 for every request; redo per request lengths)
    vc.vc_quant_kv_pack(s, max(T0), T_cap, dev(K), dev(V), *packed)
    caches = [oloop.new_draft_cache(K[b, :, :T0[b]], V[b, :, :T0[b]], bits) for b in range(B)]
    tail_k = torch.zeros((B, H, tail_cap, d), dtype=torch.int16, device=DEV)
    tail_v = torch.zeros_like(tail_k)
    tail_len = torch.zeros(B, dtype=torch.int32, device=DEV)
    packed_len = torch.tensor(T0, dtype=torch.int32, device=DEV)
    for rnd in range(12):
        kn = synth.bf16_bits(rng.standard_normal((B, k + 1, H, d)).astype(np.float32))
        vn = synth.bf16_bits(rng.standard_normal((B, k + 1, H, d)).astype(np.float32))
        n = rng.integers(0, k + 1, size=B).astype(np.int32)
        vc.vc_quant_kv_append(s, dev(kn), dev(vn), dev(n), tail_k, tail_v, tail_len, tail_cap, *packed,
                              packed_len, T_cap)
        for b in range(B):
            oloop.commit_to_draft_cache(caches[b], kn[b, :n[b] + 1].transpose(1, 0, 2),
                                        vn[b, :n[b] + 1].transpose(1, 0, 2))
    torch.cuda.synchronize()
    assert vc.vc_quant_kv_device_status() == 0
    got = to_np(packed, B, H, T_cap, d, bits)
    tl = tail_len.cpu().numpy()
    pl = packed_len.cpu().numpy()
    tk = tail_k.cpu().numpy().view(np.uint16)
    tv = tail_v.cpu().numpy().view(np.uint16)
    for b in range(B):
        c = caches[b]
        assert pl[b] == c.packed_len and tl[b] == c.tail_k.shape[1]
        want = (kivi.pack_kcodes(c.kcode, bits), kivi.pack_kmeta(c.ks, c.kz),
                kivi.pack_vcodes(c.vcode, bits), kivi.pack_vmeta(c.vs, c.vz))
        NG = c.packed_len // 32
        assert_packed_equal([g[b:b + 1, :, :NG] for g in got], want)
        assert np.array_equal(tk[b, :, :tl[b]], c.tail_k) and np.array_equal(tv[b, :, :tl[b]], c.tail_v)


def test_append_capacity_flag(vc):
    from gpu_util import DEV
    B, H, d, k = 1, 1, 64, 4
    s = vc.shape(B, H, H, d, k=k, bits=4)
    packed = alloc_packed(vc, s, 32)
    tail_k = torch.zeros((B, H, 8, d), dtype=torch.int16, device=DEV)
    tail_v = torch.zeros_like(tail_k)
    tail_len = torch.tensor([6], dtype=torch.int32, device=DEV)       # 6 + 5 > tail_cap 8
    packed_len = torch.zeros(1, dtype=torch.int32, device=DEV)
    kn = torch.zeros((B, k + 1, H, d), dtype=torch.int16, device=DEV)
    vc.vc_quant_kv_append(s, kn, kn, None, tail_k, tail_v, tail_len, 8, *packed, packed_len, 32)
    assert vc.vc_quant_kv_device_status() != 0
    assert tail_len.item() == 6 and packed_len.item() == 0            # left unchanged


def gpu_scores(vc, q, K, scale, n_obs=32):
    from gpu_util import dev, zeros_bytes, DEV
    B, Hq, _, d = q.shape
    Hkv, T = K.shape[1], K.shape[2]
    s = vc.shape(B, Hq, Hkv, d, softmax_scale=scale)
    wsb = vc.vc_token_score_workspace_size(s, T, n_obs)
    ws = zeros_bytes(wsb)
    score = torch.empty((B, Hkv, T), dtype=torch.float32, device=DEV)
    vc.vc_token_score(s, T, n_obs, dev(q), dev(K), score, ws, wsb)
    torch.cuda.synchronize()
    return score.cpu().numpy()


@pytest.mark.parametrize("B,Hq,Hkv,T,d,n_obs", [(1, 5, 1, 700, 128, 32), (2, 4, 2, 1024, 64, 32),
                                                (1, 8, 1, 333, 128, 32),
                                                (1, 1, 1, 40, 128, 16),       # one m-tile, one partial tile
                                                (1, 6, 1, 1029, 64, 32),      # 12 m-tiles, ragged 2nd range
                                                (2, 14, 2, 2100, 128, 32),    # 14 m-tiles, 3 ranges
                                                (1, 4, 1, 32, 64, 32),        # T = n_obs: row i sees i + 1 keys
                                                (32, 40, 8, 200, 128, 32),    # 256 two-tile items: q reloaded per item
                                                (4, 32, 8, 8192, 128, 32)],   # 256 items over the SMs: runs cross slices
                         ids=["g5", "g2_d64", "g8", "nr16_t40", "g6_ragged", "g7_3ranges", "t_eq_nobs",
                              "g5_many_items", "g4_runs_cross_slices"])
def test_token_score(vc, B, Hq, Hkv, T, d, n_obs):
    w = synth.get("qwen", B=B, Hq=Hq, Hkv=Hkv, T=T, d=d)
    K, _ = synth.kv(w)
    q = synth.q_obs(w, n_obs=n_obs)
    got = gpu_scores(vc, q, K, 1.0, n_obs=n_obs)
    want = tokendrop.token_scores(q, K, 1.0)
    # fp32 vs fp64.  Error budget: a log2-scaled logit carries ~1e-6 relative
    # rounding (|logit| <~ 30 -> ~3e-5 absolute), exp2 turns that into ~2e-5
    # relative on each weight, and the fp32 row sums over <= 64K keys add
    # ~3e-5 relative: 1e-3 relative leaves a 20x margin.
    err = np.abs(got - want)
    assert np.all(err <= 1e-3 * want + 1e-7 * (Hq // Hkv) * n_obs), err.max()
    assert np.allclose(got.sum(-1), (Hq // Hkv) * n_obs, rtol=1e-4)


def test_token_score_full_size_sampled(vc):
    """Qwen-32B-shaped prompt at full size (B16 Hq40 Hkv8 T65536 d128, 32
    observation queries), scored in one call with the launch the bench times (one
    persistent CTA per SM over 8192 items); sampled (request, KV head) slices
    against the fp64 oracle, with the tolerance of test_token_score."""
    w = synth.get("qwen")
    K, _ = synth.kv(w)
    q = synth.q_obs(w, n_obs=32)
    got = gpu_scores(vc, q, K, 1.0, n_obs=32)
    G = w.Hq // w.Hkv
    for (b, h) in [(0, 0), (7, 3), (w.B - 1, w.Hkv - 1)]:
        want = tokendrop.token_scores(q[b:b + 1, h * G:(h + 1) * G], K[b:b + 1, h:h + 1], 1.0)[0, 0]
        err = np.abs(got[b, h] - want)
        assert np.all(err <= 1e-3 * want + 1e-7 * G * 32), (b, h, err.max())
        assert np.isclose(got[b, h].sum(), G * 32, rtol=1e-4)


def check_selection(idx, pooled, keep, keep_last):
    """Kept set S valid: the last tokens present, ascending, and every kept candidate
    scores at least as high as every dropped one, up to 1e-4 * max(pooled): the
    GPU ranks fp32 scores (~5e-5 relative error, see test_token_score), the
    oracle fp64 ones, so a near-tie at the cut may legitimately go either way."""
    T = pooled.shape[-1]
    cand = T - keep_last
    diffs = 0
    for b in range(idx.shape[0]):
        for h in range(idx.shape[1]):
            s = idx[b, h]
            assert np.all(np.diff(s) > 0)
            assert np.array_equal(s[-keep_last:], np.arange(cand, T))
            kept = np.zeros(cand, bool)
            kept[s[:-keep_last] if keep_last else s] = True
            p = pooled[b, h, :cand]
            if kept.any() and (~kept).any():
                assert p[kept].min() >= p[~kept].max() - 1e-4 * pooled[b, h].max()
            ref = tokendrop.select_tokens(pooled[b:b + 1, h:h + 1], keep, keep_last)[0, 0]
            diffs += len(set(ref.tolist()) ^ set(s.tolist())) // 2
    return diffs


@pytest.mark.parametrize("T,keep", [(1024, 256), (4096, 1024), (160, 64)])
def test_token_select(vc, T, keep):
    from gpu_util import dev, zeros_bytes, DEV
    w = synth.get("qwen", B=2, Hq=10, Hkv=2, T=T)
    K, _ = synth.kv(w)
    q = synth.q_obs(w)
    score = gpu_scores(vc, q, K, 1.0)
    # the selection is checked against the oracle's pooled scores
    pooled = tokendrop.max_pool(tokendrop.token_scores(q, K, 1.0))
    wsb = vc.vc_token_select_workspace_size(2, 2, T)
    ws = zeros_bytes(wsb)
    idx = torch.empty((2, 2, keep), dtype=torch.int32, device=DEV)
    vc.vc_token_select(2, 2, T, dev(score.astype(np.float32)), keep, 32, 7, idx, ws, wsb)
    n_diff = check_selection(idx.cpu().numpy(), pooled, keep, 32)
    assert n_diff <= 2


def test_token_select_exact_on_given_scores(vc):
    """With the GPU's own fp32 scores as input, the selection equals the oracle's
    rule applied to those same scores, index for index (ties included)."""
    from gpu_util import dev, zeros_bytes, DEV
    rng = np.random.default_rng(1)
    B, H, T, keep = 2, 3, 2048, 512
    score = rng.integers(0, 50, size=(B, H, T)).astype(np.float32) / 7   # many ties
    wsb = vc.vc_token_select_workspace_size(B, H, T)
    ws = zeros_bytes(wsb)
    idx = torch.empty((B, H, keep), dtype=torch.int32, device=DEV)
    vc.vc_token_select(B, H, T, dev(score), keep, 32, 7, idx, ws, wsb)
    want = tokendrop.select_tokens(tokendrop.max_pool(score.astype(np.float64)), keep, 32)
    assert np.array_equal(idx.cpu().numpy(), want)
    # keep == T: identity
    idx2 = torch.empty((B, H, T), dtype=torch.int32, device=DEV)
    vc.vc_token_select(B, H, T, dev(score), T, 32, 7, idx2, ws, wsb)
    assert np.array_equal(idx2.cpu().numpy(), np.broadcast_to(np.arange(T), (B, H, T)))


def test_gather(vc):
    from gpu_util import dev, DEV
    rng = np.random.default_rng(2)
    B, H, T, d, keep = 2, 2, 300, 128, 40
    K = rng.integers(0, 2 ** 16, size=(B, H, T, d)).astype(np.uint16)
    V = rng.integers(0, 2 ** 16, size=(B, H, T, d)).astype(np.uint16)
    idx = np.sort(rng.choice(T, size=(B, H, keep)), axis=-1).astype(np.int32)
    s = vc.shape(B, H, H, d)
    Ko = torch.empty((B, H, keep, d), dtype=torch.int16, device=DEV)
    Vo = torch.empty_like(Ko)
    vc.vc_gather_kv(s, T, keep, dev(idx), dev(K), dev(V), Ko, Vo)
    assert np.array_equal(Ko.cpu().numpy().view(np.uint16), tokendrop.gather(K, idx))
    assert np.array_equal(Vo.cpu().numpy().view(np.uint16), tokendrop.gather(V, idx))
    assert vc.vc_quant_kv_device_status() == 0


def test_qwen_compressor_chain_small(vc):
    """score -> select -> gather -> 4-bit pack on a reduced Qwen-shaped layer; the
    packed result equals the oracle's quantiser applied to the same kept set."""
    from gpu_util import dev, zeros_bytes, DEV
    w = synth.get("qwen", B=2, T=2048)
    K, V = synth.kv(w)
    q = synth.q_obs(w)
    s = vc.shape(w.B, w.Hq, w.Hkv, w.d, bits=4, softmax_scale=1.0)
    keep = w.T_keep
    score = torch.empty((w.B, w.Hkv, w.T), dtype=torch.float32, device=DEV)
    wsb = vc.vc_token_score_workspace_size(s, w.T, 32)
    ws = zeros_bytes(wsb)
    Kd, Vd = dev(K), dev(V)
    vc.vc_token_score(s, w.T, 32, dev(q), Kd, score, ws, wsb)
    wsb2 = vc.vc_token_select_workspace_size(w.B, w.Hkv, w.T)
    ws2 = zeros_bytes(wsb2)
    idx = torch.empty((w.B, w.Hkv, keep), dtype=torch.int32, device=DEV)
    vc.vc_token_select(w.B, w.Hkv, w.T, score, keep, 32, 7, idx, ws2, wsb2)
    Kk = torch.empty((w.B, w.Hkv, keep, w.d), dtype=torch.int16, device=DEV)
    Vk = torch.empty_like(Kk)
    vc.vc_gather_kv(s, w.T, keep, idx, Kd, Vd, Kk, Vk)
    packed = alloc_packed(vc, s, keep)
    vc.vc_quant_kv_pack(s, keep, keep, Kk, Vk, *packed)
    torch.cuda.synchronize()
    idx_np = idx.cpu().numpy()
    pooled = tokendrop.max_pool(tokendrop.token_scores(q, K, 1.0))
    assert check_selection(idx_np, pooled, keep, 32) <= 4
    want = kivi.quant_pack(tokendrop.gather(K, idx_np), tokendrop.gather(V, idx_np), 4)
    assert_packed_equal(to_np(packed, w.B, w.Hkv, keep, w.d, 4), want)
