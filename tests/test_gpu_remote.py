"""Remote prefix caching, emulated on one GPU (VeriCache, Architecture Support,
Remote Prefix Caching): the compressed KV travels over a slow link to the GPU
that drafts, the full KV over the fast local link for verification.

A draft cache staged from a pinned "remote" store through vc_quant_kv_stage_groups
at a paced rate must equal, bit for bit, the cache packed locally, give the
same round outputs, and take at least bytes / rate to arrive.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import kivi

pytestmark = pytest.mark.gpu

W = synth.get("mistral", B=2, T=2048, k=4, V=3000, C=512)


def _group():
    from verify_compressed_kv_gb300.runtime import Group
    return Group(W.B, W.Hq, W.Hkv, W.d, W.k, W.bits, W.V, W.C, W.T, extra_tokens=8 * (W.k + 1), n_slots=2)


def _inputs():
    from verify_compressed_kv_gb300.runtime import RoundInputs

    def t(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    qd = np.stack([synth.draft_q(W, 0, i) for i in range(W.k)])[None]
    cur = [synth.draft_kv_cur(W, 0, i) for i in range(W.k)]
    kvc = np.stack([np.stack([c[j] for c in cur])[None] for j in range(2)])
    kn, vn = synth.kv_new(W, 0)
    logits, drafts, _ = synth.logits_and_drafts(W, 0)
    return RoundInputs(t(qd), t(kvc), t(synth.verify_q(W, 0)[None]), t(np.stack([kn[None], vn[None]])), t(logits),
                       t(drafts))


def test_staged_remote_prefix_equals_local_pack_and_paces_the_link():
    from verify_compressed_kv_gb300 import runtime as rt
    K, V = synth.kv(W)
    Kd = torch.from_numpy(K.view(np.int16)).cuda()
    Vd = torch.from_numpy(V.view(np.int16)).cuda()
    local = _group()
    local.load_prefix(0, Kd, Vd)
    host = local.export_packed(0, W.T)
    remote = _group()
    remote.write_store(0, Kd, Vd)                        # full KV: the fast local store
    s = torch.cuda.Stream()
    rate = 0.5                                           # GB/s, the emulated slow link
    wall = remote.stage_packed_remote(0, host, W.T, rate, s, groups_per_copy=8)
    s.synchronize()
    nbytes = sum(h.numel() * h.element_size() for h in host)
    assert nbytes == W.B * W.Hkv * W.T * 96              # 96 B per token per KV head at int2, d = 128
    assert wall >= 0.95 * nbytes / (rate * 1e9)
    ng, NGc = W.T // 32, local.P_cap // 32
    for a, b in ((local.kc, remote.kc), (local.ksz, remote.ksz), (local.vc, remote.vc), (local.vsz, remote.vsz)):
        x = a[0].view(W.B * W.Hkv, NGc, -1)[:, :ng]
        y = b[0].view(W.B * W.Hkv, NGc, -1)[:, :ng]
        assert torch.equal(x, y)
    # and the staged cache is the oracle's packing of the same K/V, bit for bit
    okc, oksz, ovc, ovsz = kivi.quant_pack(K, V, W.bits)
    for dev, want, dt in ((remote.kc, okc, np.uint32), (remote.vc, ovc, np.uint32),
                          (remote.ksz, oksz, np.float16), (remote.vsz, ovsz, np.float16)):
        got = dev[0].view(W.B * W.Hkv, NGc, -1)[:, :ng].cpu().numpy().view(dt)
        want = np.ascontiguousarray(want).reshape(W.B * W.Hkv, ng, -1)
        if dt is np.float16:
            assert np.array_equal(got.astype(np.float32), want.astype(np.float32))   # values (-0 == +0)
        else:
            assert np.array_equal(got, want.view(dt))
    assert remote.packed_len[0].tolist() == [W.T] * W.B and remote.tail_len[0].tolist() == [0] * W.B
    # one round on each: identical verify outputs and accepted lengths
    inp = _inputs()
    outs = []
    for g in (local, remote):
        cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
        tl = rt.round_single(g, inp, cs, xs)
        tl.ev["end"].synchronize()
        outs.append((g.verify_out.cpu().clone(), g.n_acc_host.clone(), g.draft_out.cpu().clone()))
        g.close()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_stage_rejects_pageable_host_memory():
    from verify_compressed_kv_gb300 import _lib as vc
    g = _group()
    host = [torch.zeros(16, dtype=torch.int32)] * 4          # not pinned
    with pytest.raises(vc.VcError) as e:
        vc.vc_quant_kv_stage_groups(g.shape, *host, 1, 0, 1, g.P_cap, g.kc[0], g.ksz[0], g.vc[0], g.vsz[0])
    assert e.value.status == 1
    g.close()
