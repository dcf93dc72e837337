"""vc_draft_attn on the GPU vs the oracle (fp64): max-abs <= 2e-2, mean-abs <= 2e-3."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import kivi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    from verify_compressed_kv_gb300 import _lib
    return _lib


def run_draft(vc, w, K, V, packed_len, tail_k, tail_v, tail_len, q, scale, k_cur=None, v_cur=None, step=0,
              T_cap=None, tail_cap=None):
    """Pack K/V on the GPU, run one draft step, return (out bf16 -> f64, tail after the call)."""
    from gpu_util import dev, zeros_bytes, bf16_to_f64, DEV
    B, H, T, d = K.shape
    T_cap = T if T_cap is None else T_cap
    tail_cap = tail_k.shape[2] if tail_cap is None else tail_cap
    s = vc.shape(B, w.Hq, H, d, bits=w.bits, softmax_scale=scale)
    kcb, kszb, vcb, vszb = vc.vc_quant_packed_bytes(s, T_cap)
    kc = torch.zeros(kcb // 4, dtype=torch.int32, device=DEV)
    ksz = torch.zeros(kszb // 2, dtype=torch.int16, device=DEV)
    vcc = torch.zeros(vcb // 4, dtype=torch.int32, device=DEV)
    vsz = torch.zeros(vszb // 2, dtype=torch.int16, device=DEV)
    vc.vc_quant_kv_pack(s, T, T_cap, dev(K), dev(V), kc, ksz, vcc, vsz)
    max_packed = int(max(packed_len))
    wsb = vc.vc_draft_attn_workspace_size(s, max_packed)
    ws = zeros_bytes(wsb)
    out = torch.empty((B, w.Hq, d), dtype=torch.int16, device=DEV)
    tk, tv = dev(tail_k), dev(tail_v)
    vc.vc_draft_attn(s, dev(q), None if k_cur is None else dev(k_cur), None if v_cur is None else dev(v_cur),
                     kc, ksz, vcc, vsz, dev(np.asarray(packed_len, np.int32)), max_packed, T_cap, tk, tv,
                     dev(np.asarray(tail_len, np.int32)), tail_cap, step, out, ws, wsb)
    torch.cuda.synchronize()
    assert vc.vc_draft_attn_device_status() == 0
    return bf16_to_f64(out), tk.cpu().numpy().view(np.uint16), tv.cpu().numpy().view(np.uint16)


CASES = [
    # name, overrides, packed_len per request, tail_len per request, step, with current token
    ("tiny", dict(), [512], [0], 0, True),
    ("tiny_tail", dict(), [480], [17], 2, True),
    ("mistral_small", dict(B=3, T=2048), [2048, 1024, 32], [0, 5, 31], 3, True),
    ("mistral_ragged_splits", dict(B=2, T=1600), [1600, 544], [1, 0], 0, False),
    ("qwen_small", dict(B=2, T=1024, keep_frac=1.0), [1024, 992], [3, 0], 1, True),
    ("llama_small", dict(B=2, T=1024, layers=1), [1024, 512], [0, 9], 0, True),
    ("g1_d64_b2", dict(B=1, Hq=2, Hkv=2, d=64, bits=2, T=640), [640], [4], 0, True),
    ("g2_d128_b4", dict(B=1, Hq=4, Hkv=2, d=128, bits=4, T=256), [256], [0], 0, True),
    ("mistral_int8", dict(B=2, T=1024, bits=8), [1024, 480], [3, 0], 1, True),
    ("g8_d64_b8", dict(B=1, Hq=8, Hkv=1, d=64, bits=8, T=320), [320], [5], 0, True),
    # G = 4 takes the transposed group product: every code width and head dim
    ("g4_d128_b4", dict(B=2, Hq=8, Hkv=2, d=128, bits=4, T=768), [768, 352], [2, 0], 1, True),
    ("g4_d64_b2", dict(B=1, Hq=4, Hkv=1, d=64, bits=2, T=512), [512], [7], 0, True),
    ("g4_d64_b8", dict(B=2, Hq=8, Hkv=2, d=64, bits=8, T=384), [384, 64], [0, 3], 2, True),
]


@pytest.mark.parametrize("name,ov,plen,tlen,step,cur", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("scale_kind", ["one", "rsqrt_d"])
def test_draft_parity(vc, name, ov, plen, tlen, step, cur, scale_kind):
    base = name.split("_")[0] if name.split("_")[0] in synth.WORKLOADS else "mistral"
    w = synth.get(base, **ov)
    scale = 1.0 if scale_kind == "one" else 1.0 / math.sqrt(w.d)
    K, V = synth.kv(w)
    rng = np.random.default_rng(len(name))
    tail_cap = 32 + w.k + 1
    tail_k = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
    tail_v = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
    q = synth.draft_q(w, 0, step)
    k_cur, v_cur = synth.draft_kv_cur(w, 0, step) if cur else (None, None)
    got, tk, tv = run_draft(vc, w, K, V, plen, tail_k, tail_v, tlen, q, scale, k_cur, v_cur, step)
    packed = kivi.quant_pack(K, V, w.bits)
    want = oatt.draft_attention(q, *packed, plen, tail_k, tail_v, tlen, w.bits, scale,
                                k_cur=k_cur, v_cur=v_cur, step=step)
    from gpu_util import assert_attn_close
    assert_attn_close(got, want, what=name)
    if cur:        # the current token was stored at tail position tail_len + step
        for b in range(w.B):
            assert np.array_equal(tk[b, :, tlen[b] + step], k_cur[b])
            assert np.array_equal(tv[b, :, tlen[b] + step], v_cur[b])


def test_draft_tail_only_equals_textbook(vc):
    """packed_len = 0: pure bf16 attention over the tail and the current token."""
    w = synth.get("mistral", B=2, T=32)
    K, V = synth.kv(w)
    rng = np.random.default_rng(0)
    tail_cap = 49
    tail_k = synth.bf16_bits(rng.standard_normal((2, 8, tail_cap, 128)).astype(np.float32))
    tail_v = synth.bf16_bits(rng.standard_normal((2, 8, tail_cap, 128)).astype(np.float32))
    q = synth.draft_q(w, 0, 0)
    got, _, _ = run_draft(vc, w, K, V, [0, 0], tail_k, tail_v, [40, 7], q, 1 / math.sqrt(128))
    G = w.G
    want = np.empty_like(got)
    for b, n in enumerate([40, 7]):
        for h in range(w.Hq):
            want[b, h] = oatt.softmax_attend(synth.bf16_to_f32(q[b, h]).astype(np.float64),
                                             synth.bf16_to_f32(tail_k[b, h // G, :n]).astype(np.float64),
                                             synth.bf16_to_f32(tail_v[b, h // G, :n]).astype(np.float64),
                                             1 / math.sqrt(128))
    from gpu_util import assert_attn_close
    assert_attn_close(got, want, what="tail only")


@pytest.mark.parametrize("name", ["mistral", "qwen", "llama", "stagger"])
def test_draft_full_size_sampled(vc, name):
    """Full-size layer (all requests, all heads in one launch, the bench's launch
    configuration); sampled (request, KV head) slices against the oracle."""
    w = synth.get(name)
    T = w.T_keep if name == "qwen" else w.T        # Qwen drafts over the kept quarter
    K, V = synth.kv(w, T=T)
    tail_cap = 32 + w.k + 1
    rng = np.random.default_rng(1)
    tlen = rng.integers(0, 32, size=w.B)
    tail_k = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
    tail_v = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
    q = synth.draft_q(w, 0, 0)
    k_cur, v_cur = synth.draft_kv_cur(w, 0, 0)
    plen = [T] * w.B
    got, _, _ = run_draft(vc, w, K, V, plen, tail_k, tail_v, tlen, q, 1.0, k_cur, v_cur, 0)
    from gpu_util import assert_attn_close
    G = w.G
    for (b, h) in [(0, 0), (w.B - 1, w.Hkv - 1), (w.B // 2, 3)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        packed = kivi.quant_pack(K[sl], V[sl], w.bits)
        want = oatt.draft_attention(q[b:b + 1, h * G:(h + 1) * G], *packed, [T], tail_k[sl], tail_v[sl],
                                    tlen[b:b + 1], w.bits, 1.0, k_cur=k_cur[sl], v_cur=v_cur[sl], step=0)
        assert_attn_close(got[b, h * G:(h + 1) * G], want[0], what=f"{name} b{b} h{h}")


def test_draft_chained_calls_equal_unchained_and_the_oracle(vc):
    """The draft steps of a round, layer after layer, as chained calls (each may
    start while the previous one finishes; one workspace shared by all): every
    output bit for bit that of the same calls each waiting for the previous, the
    tail rows each step stores, and sampled slices against the oracle with the
    tail the earlier steps wrote.  A full grid of stream CTAs (Llama-shaped
    layer, 4096 packed tokens)."""
    from gpu_util import dev, zeros_bytes, bf16_to_f64, DEV, assert_attn_close
    w = synth.get("llama", T=4096)
    L, k = 2, 3
    scale = 1.0 / math.sqrt(w.d)
    s = vc.shape(w.B, w.Hq, w.Hkv, w.d, bits=w.bits, softmax_scale=scale)
    rng = np.random.default_rng(11)
    tlen = rng.integers(0, 16, size=w.B).astype(np.int32)
    tail_cap = 32 + k + 1
    kcb, kszb, vcb, vszb = vc.vc_quant_packed_bytes(s, w.T)
    lay = []
    for l in range(L):
        K, V = synth.kv(w, layer=l)
        packed = [torch.zeros(n // e, dtype=dt, device=DEV)
                  for n, e, dt in ((kcb, 4, torch.int32), (kszb, 2, torch.int16), (vcb, 4, torch.int32), (vszb, 2, torch.int16))]
        vc.vc_quant_kv_pack(s, w.T, w.T, dev(K), dev(V), *packed)
        tk0 = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
        tv0 = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
        lay.append(dict(K=K, V=V, packed=packed, tk0=tk0, tv0=tv0))
    q = {(l, i): synth.draft_q(w, 0, i, layer=l) for l in range(L) for i in range(k)}
    cur = {(l, i): synth.draft_kv_cur(w, 0, i, layer=l) for l in range(L) for i in range(k)}
    q_d = {key: dev(v) for key, v in q.items()}
    cur_d = {key: (dev(v[0]), dev(v[1])) for key, v in cur.items()}
    plen_d, tlen_d = dev(np.full(w.B, w.T, np.int32)), dev(tlen)
    wsb = vc.vc_draft_attn_workspace_size(s, w.T)

    def run(chained):
        ws = zeros_bytes(wsb)
        tails = [(dev(x["tk0"]), dev(x["tv0"])) for x in lay]
        outs = {key: torch.empty((w.B, w.Hq, w.d), dtype=torch.int16, device=DEV) for key in q}
        torch.cuda.synchronize()
        for i in range(k):                     # nothing else on the stream between the calls
            for l in range(L):
                vc.vc_draft_attn(s, q_d[l, i], *cur_d[l, i], *lay[l]["packed"], plen_d, w.T, w.T, *tails[l], tlen_d,
                                 tail_cap, i, outs[l, i], ws, wsb,
                                 flags=vc.VC_DRAFT_CHAINED if chained and i + l > 0 else 0)
        torch.cuda.synchronize()
        assert vc.vc_draft_attn_device_status() == 0
        return ({key: o.cpu().numpy() for key, o in outs.items()},
                [(a.cpu().numpy().view(np.uint16), b.cpu().numpy().view(np.uint16)) for a, b in tails])

    plain, plain_tails = run(False)
    chained, chained_tails = run(True)
    for key in q:
        assert np.array_equal(chained[key], plain[key]), f"layer {key[0]} step {key[1]}"
    for l in range(L):
        for x, y in zip(chained_tails[l], plain_tails[l]):
            assert np.array_equal(x, y)
        for i in range(k):
            for b in range(w.B):
                assert np.array_equal(chained_tails[l][0][b, :, tlen[b] + i], cur[l, i][0][b])
                assert np.array_equal(chained_tails[l][1][b, :, tlen[b] + i], cur[l, i][1][b])
    G = w.G
    for l in range(L):
        for (b, h) in [(0, 0), (w.B - 1, w.Hkv - 1)]:
            sl = (slice(b, b + 1), slice(h, h + 1))
            pk = kivi.quant_pack(lay[l]["K"][sl], lay[l]["V"][sl], w.bits)
            tk, tv = lay[l]["tk0"][sl].copy(), lay[l]["tv0"][sl].copy()
            for i in range(k):
                want = oatt.draft_attention(q[l, i][b:b + 1, h * G:(h + 1) * G], *pk, [w.T], tk, tv, tlen[b:b + 1],
                                            w.bits, scale, k_cur=cur[l, i][0][sl], v_cur=cur[l, i][1][sl], step=i)
                got = (chained[l, i][b, h * G:(h + 1) * G].view(np.uint16).astype(np.uint32) << 16).view(np.float32)
                assert_attn_close(got.astype(np.float64), want[0], what=f"layer {l} step {i} b{b} h{h}")
                tk[0, 0, tlen[b] + i], tv[0, 0, tlen[b] + i] = cur[l, i][0][b, h], cur[l, i][1][b, h]


def test_draft_max_packed_below_capacity(vc):
    """A cache laid out for T_cap tokens holding fewer packed ones: calls with
    max_packed at the capacity and at the packed length (a different partition)
    both match the oracle, and the workspace sized for the capacity serves
    both (its size does not depend on max_packed)."""
    from gpu_util import dev, zeros_bytes, bf16_to_f64, DEV, assert_attn_close
    w = synth.get("llama", B=2, T=2048)
    T_cap, P = 4096, 2048
    scale = 1.0 / math.sqrt(w.d)
    s = vc.shape(w.B, w.Hq, w.Hkv, w.d, bits=w.bits, softmax_scale=scale)
    sizes = {mp: vc.vc_draft_attn_workspace_size(s, mp) for mp in (32, 1024, P, T_cap)}
    assert len(set(sizes.values())) == 1, sizes
    K, V = synth.kv(w)
    kcb, kszb, vcb, vszb = vc.vc_quant_packed_bytes(s, T_cap)
    packed = [torch.zeros(n // e, dtype=dt, device=DEV)
              for n, e, dt in ((kcb, 4, torch.int32), (kszb, 2, torch.int16), (vcb, 4, torch.int32), (vszb, 2, torch.int16))]
    vc.vc_quant_kv_pack(s, P, T_cap, dev(K), dev(V), *packed)
    rng = np.random.default_rng(5)
    tail_cap = 32 + w.k + 1
    tlen = np.array([3, 0], np.int32)
    tk0 = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
    tv0 = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
    q = synth.draft_q(w, 0, 0)
    k_cur, v_cur = synth.draft_kv_cur(w, 0, 0)
    plen = np.full(w.B, P, np.int32)
    want = oatt.draft_attention(q, *kivi.quant_pack(K, V, w.bits), plen, tk0, tv0, tlen, w.bits, scale,
                                k_cur=k_cur, v_cur=v_cur, step=0)
    wsb = sizes[T_cap]
    for mp in (T_cap, P):
        ws = zeros_bytes(wsb)
        out = torch.empty((w.B, w.Hq, w.d), dtype=torch.int16, device=DEV)
        vc.vc_draft_attn(s, dev(q), dev(k_cur), dev(v_cur), *packed, dev(plen), mp, T_cap, dev(tk0), dev(tv0),
                         dev(tlen), tail_cap, 0, out, ws, wsb)
        torch.cuda.synchronize()
        assert vc.vc_draft_attn_device_status() == 0
        assert_attn_close(bf16_to_f64(out), want, what=f"max_packed {mp}")


def test_draft_argument_errors(vc):
    from gpu_util import DEV
    s = vc.shape(1, 4, 1, 96, bits=2)
    with pytest.raises(vc.VcError) as e:
        vc.vc_draft_attn_workspace_size(s, 64)
    assert e.value.status == 2
    s = vc.shape(1, 4, 1, 64, bits=3)
    with pytest.raises(vc.VcError) as e:
        vc.vc_draft_attn_workspace_size(s, 64)
    assert e.value.status == 2
    s = vc.shape(1, 4, 1, 64, bits=2)
    with pytest.raises(vc.VcError) as e:
        vc.vc_draft_attn_workspace_size(s, 65)
    assert e.value.status == 1
