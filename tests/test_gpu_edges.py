"""Edge cases of the CUDA path against the oracle: empty and ragged requests,
single groups, zero-length prefixes, capacity overflow, repeat calls on one
workspace (counters must be left at zero)."""
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


def _t(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def _f64(t):
    return (t.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _pack(vc, s, K, V, T_cap):
    kcb, kszb, vcb, vszb = vc.vc_quant_packed_bytes(s, T_cap)
    arrs = [torch.zeros(kcb // 4, dtype=torch.int32, device="cuda"), torch.zeros(kszb // 2, dtype=torch.int16, device="cuda"),
            torch.zeros(vcb // 4, dtype=torch.int32, device="cuda"), torch.zeros(vszb // 2, dtype=torch.int16, device="cuda")]
    if K.shape[2]:
        vc.vc_quant_kv_pack(s, K.shape[2], T_cap, _t(K), _t(V), *arrs)
    return arrs


def test_draft_with_an_empty_request_and_repeat_calls(vc):
    """Request 1 has nothing packed and nothing in its tail: only the current token."""
    w = synth.get("mistral", B=3, T=1024)
    K, V = synth.kv(w)
    s = vc.shape(w.B, w.Hq, w.Hkv, w.d, bits=w.bits, softmax_scale=1 / math.sqrt(w.d))
    arrs = _pack(vc, s, K, V, 1024)
    tail_cap = 32 + w.k + 1
    rng = np.random.default_rng(0)
    tk = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
    tv = synth.bf16_bits(rng.standard_normal((w.B, w.Hkv, tail_cap, w.d)).astype(np.float32))
    plen, tlen = [1024, 0, 32], [3, 0, 0]
    wsb = vc.vc_draft_attn_workspace_size(s, 1024)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    packed = kivi.quant_pack(K, V, w.bits)
    for rnd in range(3):                      # repeat calls on one workspace: counters reset by the kernel
        q = synth.draft_q(w, rnd, 0)
        kc_, vc_ = synth.draft_kv_cur(w, rnd, 0)
        out = torch.empty((w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
        tkd, tvd = _t(tk), _t(tv)
        vc.vc_draft_attn(s, _t(q), _t(kc_), _t(vc_), *arrs, _t(np.array(plen, np.int32)), 1024, 1024, tkd, tvd,
                         _t(np.array(tlen, np.int32)), tail_cap, 0, out, ws, wsb)
        torch.cuda.synchronize()
        want = oatt.draft_attention(q, *packed, plen, tk, tv, tlen, w.bits, 1 / math.sqrt(w.d), k_cur=kc_, v_cur=vc_)
        err = np.abs(_f64(out) - want)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        # request 1 attends to its current token only: output = that token's V for every head
        G = w.G
        for h in range(w.Hq):
            v = synth.bf16_to_f32(vc_[1, h // G]).astype(np.float64)
            assert np.all(np.abs(_f64(out)[1, h] - v) <= 2.0 ** -8 * np.abs(v))
    assert vc.vc_draft_attn_device_status() == 0


def test_draft_wait_bound_runs_out_and_is_reported(vc):
    """Failure detection without a fault: with a short wait bound and the first
    ring stage withheld, the consumers' bounded waits run out, the call returns,
    the device status reports the barrier time-out, and the context stays usable
    (the next call, on a zeroed workspace, matches the oracle)."""
    w = synth.get("mistral", B=3, T=1024)
    K, V = synth.kv(w)
    s = vc.shape(w.B, w.Hq, w.Hkv, w.d, bits=w.bits, softmax_scale=1 / math.sqrt(w.d))
    arrs = _pack(vc, s, K, V, 1024)
    tail_cap = 32 + w.k + 1
    tk = np.zeros((w.B, w.Hkv, tail_cap, w.d), np.uint16)
    plen, tlen = [1024, 1024, 1024], [0, 0, 0]
    wsb = vc.vc_draft_attn_workspace_size(s, 1024)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    q = synth.draft_q(w, 0, 0)
    kc_, vc_ = synth.draft_kv_cur(w, 0, 0)
    assert vc.vc_draft_attn_device_status() == 0

    def call():
        out = torch.empty((w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
        vc.vc_draft_attn(s, _t(q), _t(kc_), _t(vc_), *arrs, _t(np.array(plen, np.int32)), 1024, 1024, _t(tk), _t(tk),
                         _t(np.array(tlen, np.int32)), tail_cap, 0, out, ws, wsb)
        torch.cuda.synchronize()
        return out

    try:
        vc.vc_draft_attn_test_hooks(2_000_000, 1)          # ~1 ms per wait, first stage withheld
        call()
        status = vc.vc_draft_attn_device_status()
    finally:
        vc.vc_draft_attn_test_hooks(0, 0)
    assert status & 1, f"barrier time-out not reported (status {status})"
    ws.zero_()                                               # the timed-out call left its counters
    out = call()
    want = oatt.draft_attention(q, *kivi.quant_pack(K, V, w.bits), plen, tk, tk, tlen, w.bits, 1 / math.sqrt(w.d),
                                k_cur=kc_, v_cur=vc_)
    err = np.abs(_f64(out) - want)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert vc.vc_draft_attn_device_status() == 0


def test_draft_test_hooks_reject_bad_arguments(vc):
    with pytest.raises(vc.VcError):
        vc.vc_draft_attn_test_hooks(10, 0)
    with pytest.raises(vc.VcError):
        vc.vc_draft_attn_test_hooks(0, 2)
    vc.vc_draft_attn_test_hooks(0, 0)


def test_draft_single_group_and_no_current_token(vc):
    w = synth.get("qwen", B=1, T=32, keep_frac=1.0)
    K, V = synth.kv(w)
    s = vc.shape(1, w.Hq, w.Hkv, w.d, bits=w.bits, softmax_scale=1.0)
    arrs = _pack(vc, s, K, V, 32)
    tail_cap = 4
    tk = np.zeros((1, w.Hkv, tail_cap, w.d), np.uint16)
    wsb = vc.vc_draft_attn_workspace_size(s, 32)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    q = synth.draft_q(w, 0, 0)
    out = torch.empty((1, w.Hq, w.d), dtype=torch.int16, device="cuda")
    vc.vc_draft_attn(s, _t(q), None, None, *arrs, _t(np.array([32], np.int32)), 32, 32, _t(tk), _t(tk),
                     _t(np.array([0], np.int32)), tail_cap, 0, out, ws, wsb)
    torch.cuda.synchronize()
    want = oatt.draft_attention(q, *kivi.quant_pack(K, V, w.bits), [32], tk, tk, [0], w.bits, 1.0)
    err = np.abs(_f64(out) - want)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_pack_zero_tokens_is_a_no_op(vc):
    s = vc.shape(2, 4, 2, 64, bits=4)
    kcb, kszb, vcb, vszb = vc.vc_quant_packed_bytes(s, 64)
    kc = torch.full((kcb // 4,), 7, dtype=torch.int32, device="cuda")
    z = torch.zeros(16, dtype=torch.int16, device="cuda")
    vc.vc_quant_kv_pack(s, 0, 64, z, z, kc, z, kc, z)
    torch.cuda.synchronize()
    assert int((kc != 7).sum()) == 0


def test_verify_commit_capacity_overflow_is_flagged_and_leaves_state(vc):
    w = synth.get("mistral", B=2, T=256, k=3)
    s = vc.shape(w.B, w.Hq, w.Hkv, w.d, k=w.k)
    C, T_cap = 128, 256
    host = torch.zeros(T_cap // C * 2 * w.B * w.Hkv * C * w.d, dtype=torch.int16).pin_memory()
    before = host.clone()
    plen = torch.tensor([254, 10], dtype=torch.int32, device="cuda")     # request 0: 254 + 4 > 256
    kn, vn = synth.kv_new(w, 0)
    n_acc = torch.tensor([3, 0], dtype=torch.int32, device="cuda")
    vc.vc_verify_commit(s, _t(kn), _t(vn), n_acc, plen, host, C, T_cap)
    torch.cuda.synchronize()
    assert vc.vc_verify_attn_device_status() != 0
    p = plen.cpu().numpy()
    assert p[0] == 254 and p[1] == 11                          # request 0 untouched, request 1 committed
    st = host.numpy().view(np.uint16).reshape(T_cap // C, 2, w.B, w.Hkv, C, w.d)
    st0 = before.numpy().view(np.uint16).reshape(T_cap // C, 2, w.B, w.Hkv, C, w.d)
    assert np.array_equal(st[:, :, 0], st0[:, :, 0])
    assert np.array_equal(st[0, 0, 1, :, 10], kn[1, 0]) and np.array_equal(st[0, 1, 1, :, 10], vn[1, 0])


def test_verify_zero_prefix_equals_new_tokens_only(vc):
    """No prefix at all (a request's first verification): rows attend to new tokens only."""
    w = synth.get("mistral", B=1, T=0, k=5)
    s = vc.shape(1, w.Hq, w.Hkv, w.d, k=w.k, softmax_scale=1.0)
    q = synth.verify_q(w, 0)
    kn, vn = synth.kv_new(w, 0)
    wsb = vc.vc_verify_attn_workspace_size(s, 1)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    out = torch.empty((1, w.k + 1, w.Hq, w.d), dtype=torch.int16, device="cuda")
    vc.vc_verify_attn_finish(s, _t(q), _t(kn), _t(vn), 1, False, out, ws, wsb)
    torch.cuda.synchronize()
    want = oatt.verify_attention(q, np.zeros((1, w.Hkv, 0, w.d), np.uint16), np.zeros((1, w.Hkv, 0, w.d), np.uint16),
                                 kn, vn, [0], 1.0)
    err = np.abs(_f64(out) - want)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    # row 0 sees only new token 0: output = v_new[0]
    G = w.G
    for h in range(w.Hq):
        v = synth.bf16_to_f32(vn[0, 0, h // G]).astype(np.float64)
        assert np.all(np.abs(_f64(out)[0, 0, h] - v) <= 2.0 ** -8 * np.abs(v))
