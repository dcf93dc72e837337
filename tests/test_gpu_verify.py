"""vc_verify_attn on the GPU vs the oracle (fp64), the streamed pipeline and commit."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    from verify_compressed_kv_gb300 import _lib
    return _lib


def host_store(K, V, C, n_chunks):
    """[B,H,T,d] K/V -> chunk-major [n_chunks, 2, B, H, C, d] (bf16 bits), zero padded."""
    B, H, T, d = K.shape
    st = np.zeros((n_chunks, 2, B, H, C, d), np.uint16)
    for c in range((T + C - 1) // C):
        n = min(C, T - c * C)
        st[c, 0, :, :, :n] = K[:, :, c * C:c * C + n]
        st[c, 1, :, :, :n] = V[:, :, c * C:c * C + n]
    return st


def run_lowlevel(vc, w, K, V, q, kn, vn, plen, C, parts, scale):
    """Chunks already on the device: vc_verify_attn_chunk per chunk + finish."""
    from gpu_util import dev, zeros_bytes, bf16_to_f64, DEV
    B, H, T, d = K.shape
    s = vc.shape(B, w.Hq, H, d, k=w.k, softmax_scale=scale)
    n_chunks = (max(plen) + C - 1) // C
    st = host_store(K, V, C, max(n_chunks, 1))
    wsb = vc.vc_verify_attn_workspace_size(s, parts)
    ws = zeros_bytes(wsb)
    out = torch.empty((B, w.k + 1, w.Hq, d), dtype=torch.int16, device=DEV)
    qd, pl = dev(q), dev(np.asarray(plen, np.int32))
    for c in range(n_chunks):
        vc.vc_verify_attn_chunk(s, qd, dev(st[c]), C, c * C, pl, parts, c == 0, ws, wsb)
    vc.vc_verify_attn_finish(s, qd, dev(kn), dev(vn), parts, n_chunks > 0, out, ws, wsb)
    torch.cuda.synchronize()
    return bf16_to_f64(out)


CASES = [
    ("tiny", dict(), 128, 1, [512]),
    ("tiny_parts", dict(), 128, 3, [512]),
    ("mistral_small", dict(B=3, T=3000, k=16), 1024, 2, [3000, 1500, 1]),
    ("qwen_small", dict(B=2, T=1100, k=32), 512, 1, [1100, 1024]),
    ("llama_small", dict(B=2, T=777, k=32, layers=1), 256, 4, [777, 0]),
    ("stagger_small", dict(B=2, T=640, k=24), 256, 2, [640, 639]),
    ("g1_d64", dict(B=1, Hq=2, Hkv=2, d=64, T=300, k=3), 128, 2, [300]),
]


@pytest.mark.parametrize("name,ov,C,parts,plen", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("scale_kind", ["one", "rsqrt_d"])
def test_verify_parity(vc, name, ov, C, parts, plen, scale_kind):
    base = name.split("_")[0] if name.split("_")[0] in synth.WORKLOADS else "mistral"
    w = synth.get(base, **ov)
    scale = 1.0 if scale_kind == "one" else 1.0 / math.sqrt(w.d)
    K, V = synth.kv(w)
    q = synth.verify_q(w, 0)
    kn, vn = synth.kv_new(w, 0)
    got = run_lowlevel(vc, w, K, V, q, kn, vn, plen, C, parts, scale)
    want = oatt.verify_attention(q, K, V, kn, vn, plen, scale)
    from gpu_util import assert_attn_close
    assert_attn_close(got, want, what=name)


def test_verify_causality_bitwise(vc):
    """Changing new tokens after j leaves rows 0..j bit-for-bit unchanged."""
    w = synth.get("mistral", B=2, T=700, k=6)
    K, V = synth.kv(w)
    q = synth.verify_q(w, 0)
    kn, vn = synth.kv_new(w, 0)
    a = run_lowlevel(vc, w, K, V, q, kn, vn, [700, 650], 256, 2, 1.0)
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[:, 4:] ^= np.uint16(0x5A5A)
    vn2[:, 4:] ^= np.uint16(0x1234)
    b = run_lowlevel(vc, w, K, V, q, kn2, vn2, [700, 650], 256, 2, 1.0)
    assert np.array_equal(a[:, :4], b[:, :4])
    assert not np.array_equal(a[:, 4:], b[:, 4:])


def test_verify_row_equals_k0_decode(vc):
    """Row j of a k-row verify equals a k=0 verify (decode) at prefix T + j
    (within tolerance: different reduction order)."""
    w = synth.get("mistral", B=1, T=512, k=5)
    K, V = synth.kv(w)
    q = synth.verify_q(w, 0)
    kn, vn = synth.kv_new(w, 0)
    full = run_lowlevel(vc, w, K, V, q, kn, vn, [512], 128, 1, 1.0)
    from gpu_util import assert_attn_close
    for j in range(w.k + 1):
        Kj = np.concatenate([K, kn[:, :j].transpose(0, 2, 1, 3)], axis=2)
        Vj = np.concatenate([V, vn[:, :j].transpose(0, 2, 1, 3)], axis=2)
        w0 = synth.get("mistral", B=1, T=512 + j, k=0)
        dec = run_lowlevel(vc, w0, Kj, Vj, q[:, j:j + 1], kn[:, j:j + 1], vn[:, j:j + 1], [512 + j], 128, 1, 1.0)
        assert_attn_close(full[:, j], dec[:, 0], max_abs=1e-2, mean_abs=1e-3, what=f"row {j}")


def test_streamed_pipeline_and_commit(vc):
    """Pinned host store -> ring of device slots (copy stream) -> chunk kernels
    (compute stream); then commit of accepted rows into the host store."""
    from gpu_util import dev, zeros_bytes, bf16_to_f64, pinned, DEV
    w = synth.get("mistral", B=3, T=2500, k=8)
    C, parts, n_slots = 512, 2, 2
    K, V = synth.kv(w)
    T_cap = 4096
    n_chunks_cap = T_cap // C
    st = pinned(host_store(K, V, C, n_chunks_cap))
    plen = np.array([2500, 1800, 2048], np.int32)
    s = vc.shape(w.B, w.Hq, w.Hkv, w.d, k=w.k, softmax_scale=1 / math.sqrt(w.d))
    slot_elems = 2 * w.B * w.Hkv * C * w.d
    slots = torch.empty(n_slots * slot_elems, dtype=torch.int16, device=DEV)
    wsb = vc.vc_verify_attn_workspace_size(s, parts)
    ws = zeros_bytes(wsb)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    pipe = vc.vc_verify_pipeline_create(n_slots)
    try:
        from gpu_util import assert_attn_close
        pl = dev(plen)
        for rnd in range(3):
            q = synth.verify_q(w, rnd)
            kn, vn = synth.kv_new(w, rnd)
            out = torch.empty((w.B, w.k + 1, w.Hq, w.d), dtype=torch.int16, device=DEV)
            qd, knd, vnd = dev(q), dev(kn), dev(vn)
            torch.cuda.synchronize()
            max_prefix = int(plen.max())
            vc.vc_verify_prefetch(pipe, s, st, C, max_prefix, T_cap, slots, xs)
            vc.vc_verify_attn_streamed(pipe, s, qd, st, C, max_prefix, T_cap, pl, slots, knd, vnd, out, parts, ws, wsb,
                                       cs, xs)
            cs.synchronize()
            Kcur = np.zeros((w.B, w.Hkv, T_cap, w.d), np.uint16)
            Vcur = np.zeros_like(Kcur)
            host = st.numpy().view(np.uint16)
            for c in range(n_chunks_cap):
                Kcur[:, :, c * C:(c + 1) * C] = host[c, 0]
                Vcur[:, :, c * C:(c + 1) * C] = host[c, 1]
            want = oatt.verify_attention(q, Kcur, Vcur, kn, vn, plen, 1 / math.sqrt(w.d))
            assert_attn_close(bf16_to_f64(out), want, what=f"round {rnd}")
            # accept a few rows and commit them to the host store
            n_acc = np.array([rnd, w.k, 0], np.int32)
            with torch.cuda.stream(cs):
                vc.vc_verify_commit(s, knd, vnd, dev(n_acc), pl, st, C, T_cap, cs)
            cs.synchronize()
            for b in range(w.B):
                for r in range(n_acc[b] + 1):
                    pos = plen[b] + r
                    c, t = divmod(pos, C)
                    assert np.array_equal(host[c, 0, b, :, t], kn[b, r])
                    assert np.array_equal(host[c, 1, b, :, t], vn[b, r])
            plen = plen + n_acc + 1
            assert np.array_equal(pl.cpu().numpy(), plen)
        assert vc.vc_verify_attn_device_status() == 0
    finally:
        vc.vc_verify_pipeline_destroy(pipe)


def test_streamed_rejects_pageable_host_memory(vc):
    from gpu_util import zeros_bytes, DEV
    s = vc.shape(1, 4, 1, 64, k=1)
    pipe = vc.vc_verify_pipeline_create(1)
    try:
        host = torch.zeros(2 * 64 * 64, dtype=torch.int16)      # not pinned
        with pytest.raises(vc.VcError) as e:
            vc.vc_verify_prefetch(pipe, s, host, 64, 64, 64, torch.empty(8192, dtype=torch.int16, device=DEV), None)
        assert e.value.status == 1
    finally:
        vc.vc_verify_pipeline_destroy(pipe)


@pytest.mark.parametrize("name", ["mistral", "qwen", "llama", "stagger"])
def test_verify_full_size_sampled(vc, name):
    """Full-size prefix, every request and head in the bench's launch
    configuration (chunks of 4096, streamed); sampled (request, KV head)
    slices against the oracle."""
    from gpu_util import dev, zeros_bytes, bf16_to_f64, pinned, DEV, assert_attn_close
    w = synth.get(name)
    K, V = synth.kv(w)
    C, n_slots = w.C, 2
    n_chunks = w.T // C
    st = pinned(host_store(K, V, C, n_chunks))
    s = vc.shape(w.B, w.Hq, w.Hkv, w.d, k=w.k, softmax_scale=1.0)
    parts = vc.vc_verify_attn_parts(s, C)                   # as the runtime plans it
    assert 1 <= parts <= 16
    slots = torch.empty(n_slots * 2 * w.B * w.Hkv * C * w.d, dtype=torch.int16, device=DEV)
    wsb = vc.vc_verify_attn_workspace_size(s, parts)
    ws = zeros_bytes(wsb)
    q = synth.verify_q(w, 0)
    kn, vn = synth.kv_new(w, 0)
    out = torch.empty((w.B, w.k + 1, w.Hq, w.d), dtype=torch.int16, device=DEV)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    pipe = vc.vc_verify_pipeline_create(n_slots)
    try:
        qd, knd, vnd = dev(q), dev(kn), dev(vn)
        pl = dev(np.full(w.B, w.T, np.int32))
        torch.cuda.synchronize()
        vc.vc_verify_attn_streamed(pipe, s, qd, st, C, w.T, n_chunks * C, pl, slots, knd, vnd, out, parts, ws, wsb, cs, xs)
        cs.synchronize()
    finally:
        vc.vc_verify_pipeline_destroy(pipe)
    got = bf16_to_f64(out)
    G = w.G
    for (b, h) in [(0, 0), (w.B - 1, w.Hkv - 1)]:
        want = oatt.verify_attention(q[b:b + 1, :, h * G:(h + 1) * G], K[b:b + 1, h:h + 1], V[b:b + 1, h:h + 1],
                                     kn[b:b + 1, :, h:h + 1], vn[b:b + 1, :, h:h + 1], [w.T], 1.0)
        assert_attn_close(got[b:b + 1, :, h * G:(h + 1) * G], want, what=f"{name} b{b} h{h}")
