"""Cross-resource staggering must not change results (VeriCache, Technical
Summary, Key System Innovations (1): the staggered schedule overlaps one
group's drafting with another group's verification transfer instead of
running all drafts then all verifications in lock-step).

Two request groups run the same per-group sequence of (draft cycle i, verify
cycle i) under both schedules; every verify output, accepted length, the
packed draft caches, the tails and the pinned full-KV stores must be
bit-identical.  One verify output is also checked against the oracle.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt

pytestmark = pytest.mark.gpu

W = synth.get("stagger", B=3, T=1536, k=6, V=3000, C=512)
N_CYCLES = 3


def inputs(gi, cyc):
    from verify_compressed_kv_gb300.runtime import RoundInputs

    def t(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    qd = np.stack([synth.draft_q(W, cyc, i, 0, gi) for i in range(W.k)])[None]
    cur = [synth.draft_kv_cur(W, cyc, i, 0, gi) for i in range(W.k)]
    kvc = np.stack([np.stack([c[j] for c in cur])[None] for j in range(2)])
    qv = synth.verify_q(W, cyc, 0, gi)[None]
    kn, vn = synth.kv_new(W, cyc, 0, gi)
    logits, drafts, _ = synth.logits_and_drafts(W, cyc, gi)
    return RoundInputs(t(qd), t(kvc), t(qv), t(np.stack([kn[None], vn[None]])), t(logits), t(drafts))


def build():
    from verify_compressed_kv_gb300.runtime import Group
    gs = []
    for gi in range(2):
        g = Group(W.B, W.Hq, W.Hkv, W.d, W.k, W.bits, W.V, W.C, W.T, extra_tokens=(N_CYCLES + 2) * (W.k + 1),
                  n_slots=2)
        K, V = synth.kv(W, group=gi)
        g.load_prefix(0, torch.from_numpy(K.view(np.int16)).cuda(), torch.from_numpy(V.view(np.int16)).cuda())
        gs.append(g)
    torch.cuda.synchronize()
    return gs


def state(g):
    """Draft cache, tail, lengths and the committed part of the full-KV store
    (capacity beyond each request's prefix was never written)."""
    out = [x.cpu().numpy().copy() for x in (g.kc[0], g.ksz[0], g.vc[0], g.vsz[0], g.packed_len[0], g.tail_len[0],
                                            g.prefix_len[0])]
    tl = g.tail_len[0].cpu().numpy()
    tk, tv = g.tail_k[0].cpu().numpy(), g.tail_v[0].cpu().numpy()
    out += [tk[b, :, :tl[b]].copy() for b in range(g.B)] + [tv[b, :, :tl[b]].copy() for b in range(g.B)]
    st = g.host_kv[0].numpy().reshape(g.n_chunks_cap, 2, g.B, g.Hkv, g.C, g.d)
    full = st.transpose(1, 2, 3, 0, 4, 5).reshape(2, g.B, g.Hkv, g.n_chunks_cap * g.C, g.d)
    pl = g.prefix_len[0].cpu().numpy()
    out += [full[:, b, :, :pl[b]].copy() for b in range(g.B)]
    return out


def run(schedule):
    from verify_compressed_kv_gb300 import runtime as rt
    groups = build()
    inp = [[inputs(gi, c) for c in range(N_CYCLES)] for gi in range(2)]
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    outs = {0: [], 1: []}
    nacc = {0: [], 1: []}
    if schedule == "lockstep":
        for c in range(N_CYCLES):
            tl = rt.round_lockstep(groups, [inp[0][c], inp[1][c]], cs, xs)
            tl.ev["end"].synchronize()
            for gi, g in enumerate(groups):
                outs[gi].append(g.verify_out.cpu().numpy().copy())
                nacc[gi].append(g.n_acc_host.numpy().copy())
                g.after_round()
    else:
        for r in range(2 * N_CYCLES + 1):
            X, Y = groups[r % 2], groups[(r + 1) % 2]
            xi, yi = r % 2, (r + 1) % 2
            dc, vcyc = r // 2, (r - 1) // 2
            if r == 0:                          # prologue: group 0 drafts its first cycle
                for i in range(X.k):
                    X.draft_step(inp[xi][0], 0, i, cs)
                cs.synchronize()
                continue
            if dc >= N_CYCLES:                  # epilogue: only the verification is left
                tl = rt.Timeline()
                tl.mark("start", cs)
                for l in range(Y.L):
                    Y.verify(inp[yi][vcyc], l, cs, xs)
                Y.accept(inp[yi][vcyc], cs)
                Y.commit(inp[yi][vcyc], cs)
                Y.read_back(cs)
                tl.mark("end", cs)
            else:
                tl = rt.round_staggered(X, Y, inp[xi][dc], inp[yi][vcyc], cs, xs)
            tl.ev["end"].synchronize()
            outs[yi].append(Y.verify_out.cpu().numpy().copy())
            nacc[yi].append(Y.n_acc_host.numpy().copy())
            Y.after_round()
    st = [state(g) for g in groups]
    for g in groups:
        g.close()
    return outs, nacc, st


def test_staggered_equals_lockstep():
    o_s, n_s, st_s = run("staggered")
    o_l, n_l, st_l = run("lockstep")
    for gi in range(2):
        assert len(n_s[gi]) == N_CYCLES and len(n_l[gi]) == N_CYCLES
        for c in range(N_CYCLES):
            assert np.array_equal(n_s[gi][c], n_l[gi][c])
            assert np.array_equal(o_s[gi][c], o_l[gi][c]), f"group {gi} cycle {c} verify output differs"
        for a, b in zip(st_s[gi], st_l[gi]):
            assert np.array_equal(a, b)


def test_first_verify_against_oracle():
    o_s, _, _ = run("staggered")
    q = synth.verify_q(W, 0, 0, 1)
    kn, vn = synth.kv_new(W, 0, 0, 1)
    K, V = synth.kv(W, group=1)
    G = W.G
    got = (o_s[1][0].view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    b, h = 1, 5
    want = oatt.verify_attention(q[b:b + 1, :, h * G:(h + 1) * G], K[b:b + 1, h:h + 1], V[b:b + 1, h:h + 1],
                                 kn[b:b + 1, :, h:h + 1], vn[b:b + 1, :, h:h + 1], [W.T], 1.0)
    err = np.abs(got[b:b + 1, :, h * G:(h + 1) * G] - want)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_inputs_arriving_on_another_stream():
    """round_single with `ready`: the round's inputs copied from pinned host
    memory on their own stream while the full-KV transfer starts; the results
    equal a round on device-resident inputs."""
    from verify_compressed_kv_gb300 import runtime as rt
    from verify_compressed_kv_gb300.runtime import RoundInputs
    cs, xs, ins = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    res = []
    for mode in ("resident", "copied"):
        g, other = build()
        other.close()
        outs = []
        for c in range(N_CYCLES):
            inp = inputs(0, c)
            ready = None
            if mode == "copied":
                host = RoundInputs(*[getattr(inp, n).cpu().pin_memory() for n in
                                     ("q_draft", "kv_cur", "q_verify", "kv_new", "logits", "drafts")])
                dst = RoundInputs(*[torch.empty_like(getattr(inp, n)) for n in
                                    ("q_draft", "kv_cur", "q_verify", "kv_new", "logits", "drafts")])
                torch.cuda.synchronize()
                with torch.cuda.stream(ins):
                    for n in ("q_draft", "kv_cur", "q_verify", "kv_new", "logits", "drafts"):
                        getattr(dst, n).copy_(getattr(host, n), non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(ins)
                inp = dst
            tl = rt.round_single(g, inp, cs, xs, ready=ready)
            tl.ev["end"].synchronize()
            outs.append((g.verify_out.cpu().numpy().copy(), g.n_acc.cpu().numpy().copy(),
                         g.next_tok.cpu().numpy().copy()))
            g.after_round()
        res.append(outs + [state(g)])
        g.close()
    for a, b in zip(res[0][:-1], res[1][:-1]):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
    for x, y in zip(res[0][-1], res[1][-1]):
        assert np.array_equal(x, y)
