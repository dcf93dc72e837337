"""The draft -> verify -> accept loop over the C ABI, for one request.

VeriCache (gist.science/paper/2605.17613), Technical Summary, Core Algorithm:
draft k tokens with the compressed KV, verify them in one forward pass with
the full KV, keep them up to the first disagreement plus the full-KV token
there, and continue from the last kept token.  Architecture Support: the
compressed KV stays in GPU memory, the full KV in pinned host memory and is
streamed to the GPU for every verification.

The model is anything with ``forward(tokens, positions, attend)`` returning
(logits [n, V], per-layer K and V [n, Hkv, d] as bf16 bits) and calling
``attend(layer, q, k, v)`` once per layer (q [n, Hq, d], k/v [n, Hkv, d],
bf16 bits as numpy uint16) for the attention output.  Everything outside
attention is the model's; every attention, accept and commit step runs in the
CUDA libraries.

Draft-cache bookkeeping: draft step i stores the current token's K/V at tail
position tail_len + i (vc_draft_attn does it); after accept, the exact K/V of
the n+1 kept tokens (the verify pass's) replace them (vc_quant_kv_append) and
go to the full-KV store (vc_verify_commit).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import _lib as vc

GROUP = 32


def _dev(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def _bf16_out(t: torch.Tensor) -> np.ndarray:
    u = t.cpu().numpy().view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


class _Layer:
    """Device / pinned state of one attention layer for one request."""

    def __init__(self, sh, C, T_cap, P_cap, tail_cap, n_slots, device):
        self.sh = sh
        Hkv, d = sh.Hkv, sh.d
        self.C = C
        self.T_cap = T_cap
        self.P_cap = P_cap
        self.tail_cap = tail_cap
        kcb, kszb, vcb, vszb = vc.vc_quant_packed_bytes(sh, P_cap)
        self.kc = torch.zeros(kcb // 4, dtype=torch.int32, device=device)
        self.ksz = torch.zeros(kszb // 2, dtype=torch.int16, device=device)
        self.vc = torch.zeros(vcb // 4, dtype=torch.int32, device=device)
        self.vsz = torch.zeros(vszb // 2, dtype=torch.int16, device=device)
        self.tail_k = torch.zeros((1, Hkv, tail_cap, d), dtype=torch.int16, device=device)
        self.tail_v = torch.zeros_like(self.tail_k)
        self.packed_len = torch.zeros(1, dtype=torch.int32, device=device)
        self.tail_len = torch.zeros(1, dtype=torch.int32, device=device)
        self.chunk_elems = 2 * Hkv * C * d
        self.host = torch.zeros((T_cap // C) * self.chunk_elems, dtype=torch.int16, pin_memory=True)
        self.prefix_len = torch.zeros(1, dtype=torch.int32, device=device)
        self.slots = torch.empty(n_slots * self.chunk_elems, dtype=torch.int16, device=device)


class GpuSpeculativeDecoder:
    """Draft/verify/accept decoding of one request on the GPU (B = 1)."""

    def __init__(self, n_layers, Hq, Hkv, d, vocab, k, bits, scale, C=128, max_tokens=4096, n_slots=4,
                 device="cuda"):
        self.L, self.k, self.V = n_layers, k, vocab
        self.device = torch.device(device)
        self.scale = scale
        self.sh = vc.shape(1, Hq, Hkv, d, k=k, bits=bits, softmax_scale=scale)
        self.sh0 = vc.shape(1, Hq, Hkv, d, k=0, bits=bits, softmax_scale=scale)
        self.T_cap = int(math.ceil(max_tokens / C) * C)
        self.P_cap = int(math.ceil(max_tokens / GROUP) * GROUP)
        self.tail_cap = GROUP + k + 1
        self.layers = [_Layer(self.sh, C, self.T_cap, self.P_cap, self.tail_cap, n_slots, self.device)
                       for _ in range(n_layers)]
        self.max_prefix = 0
        self.pipe = vc.vc_verify_pipeline_create(n_slots)
        self.cs = torch.cuda.Stream(self.device)
        self.xs = torch.cuda.Stream(self.device)
        self.ws_draft_bytes = vc.vc_draft_attn_workspace_size(self.sh, self.P_cap)
        self.ws_draft = torch.zeros(self.ws_draft_bytes, dtype=torch.uint8, device=self.device)
        self.ws_v_bytes = vc.vc_verify_attn_workspace_size(self.sh, 1)
        self.ws_v = torch.zeros(self.ws_v_bytes, dtype=torch.uint8, device=self.device)
        self.ws_a_bytes = max(vc.vc_accept_workspace_size(1, kk, vocab) for kk in range(1, k + 1))
        self.ws_a = torch.zeros(self.ws_a_bytes, dtype=torch.uint8, device=self.device)
        self.k_new = [None] * n_layers
        self.v_new = [None] * n_layers

    def close(self):
        if self.pipe:
            vc.vc_verify_pipeline_destroy(self.pipe)
            self.pipe = None

    # ------------------------------------------------------------ prefill
    def load_prompt(self, K_layers, V_layers, draft_K=None, draft_V=None):
        """Full prefix K/V per layer ([Hkv, T, d] bf16 bits) -> pinned store; the
        draft cache gets whole 32-groups packed, the rest in the tail.  draft_K /
        draft_V optionally replace the tokens the draft cache is built from
        (token dropping)."""
        for li, lay in enumerate(self.layers):
            K, V = K_layers[li], V_layers[li]
            Hkv, T, d = K.shape
            st = lay.host.view(self.T_cap // lay.C, 2, 1, Hkv, lay.C, d)
            Kt = torch.from_numpy(np.ascontiguousarray(K).view(np.int16))
            Vt = torch.from_numpy(np.ascontiguousarray(V).view(np.int16))
            for c in range((T + lay.C - 1) // lay.C):
                n = min(lay.C, T - c * lay.C)
                st[c, 0, 0, :, :n].copy_(Kt[:, c * lay.C:c * lay.C + n])
                st[c, 1, 0, :, :n].copy_(Vt[:, c * lay.C:c * lay.C + n])
            lay.prefix_len.fill_(T)
            dK = K if draft_K is None else draft_K[li]
            dV = V if draft_V is None else draft_V[li]
            P = (dK.shape[1] // GROUP) * GROUP
            if P:
                vc.vc_quant_kv_pack(self.sh, P, self.P_cap, _dev(dK[None, :, :P], self.device),
                                    _dev(dV[None, :, :P], self.device), lay.kc, lay.ksz, lay.vc, lay.vsz, self.cs)
            rest = dK.shape[1] - P
            if rest:
                lay.tail_k[0, :, :rest].copy_(_dev(dK[:, P:], self.device))
                lay.tail_v[0, :, :rest].copy_(_dev(dV[:, P:], self.device))
            lay.packed_len.fill_(P)
            lay.tail_len.fill_(rest)
            self.max_prefix = T
        torch.cuda.synchronize(self.device)

    # ------------------------------------------------------------ attention steps
    def draft_attend(self, layer, q, k, v, step):
        lay = self.layers[layer]
        out = torch.empty((1, self.sh.Hq, self.sh.d), dtype=torch.int16, device=self.device)
        vc.vc_draft_attn(self.sh, _dev(q, self.device), _dev(k, self.device), _dev(v, self.device),
                         lay.kc, lay.ksz, lay.vc, lay.vsz, lay.packed_len, self.P_cap, self.P_cap,
                         lay.tail_k, lay.tail_v, lay.tail_len, self.tail_cap, step, out, self.ws_draft,
                         self.ws_draft_bytes, self.cs)
        self.cs.synchronize()
        return _bf16_out(out)

    def verify_attend(self, layer, q, k, v, sh=None):
        """Rows = the new tokens (k+1 for verify, 1 for plain decoding)."""
        sh = sh or self.sh
        lay = self.layers[layer]
        n = q.shape[0]
        out = torch.empty((1, n, sh.Hq, sh.d), dtype=torch.int16, device=self.device)
        kn, vn = _dev(k[None], self.device), _dev(v[None], self.device)
        self.k_new[layer], self.v_new[layer] = kn, vn
        ws_bytes = vc.vc_verify_attn_workspace_size(sh, 1)
        ws = self.ws_v if ws_bytes <= self.ws_v_bytes else torch.zeros(ws_bytes, dtype=torch.uint8,
                                                                        device=self.device)
        vc.vc_verify_attn_streamed(self.pipe, sh, _dev(q[None], self.device), lay.host, lay.C, self.max_prefix,
                                   lay.T_cap, lay.prefix_len, lay.slots, kn, vn, out, 1, ws, ws.numel(), self.cs,
                                   self.xs)
        self.cs.synchronize()
        return _bf16_out(out)[0]

    def accept(self, logits, drafts):
        lg = torch.from_numpy(np.ascontiguousarray(logits[None], np.float32)).to(self.device)
        dr = torch.from_numpy(np.ascontiguousarray(np.asarray(drafts, np.int32)[None])).to(self.device)
        n = torch.empty(1, dtype=torch.int32, device=self.device)
        nxt = torch.empty(1, dtype=torch.int32, device=self.device)
        vc.vc_accept(1, len(drafts), self.V, lg, dr, n, nxt, None, self.ws_a, self.ws_a_bytes, self.cs)
        self.cs.synchronize()
        return int(n.item()), int(nxt.item())

    def commit(self, n_acc, sh=None, append_draft=True):
        """Kept rows 0..n_acc of the last verify pass -> full-KV store (+ draft cache)."""
        sh = sh or self.sh
        n_t = torch.tensor([n_acc], dtype=torch.int32, device=self.device)
        for li, lay in enumerate(self.layers):
            vc.vc_verify_commit(sh, self.k_new[li], self.v_new[li], n_t, lay.prefix_len, lay.host, lay.C,
                                self.T_cap, self.cs)
            if append_draft:
                vc.vc_quant_kv_append(sh, self.k_new[li], self.v_new[li], n_t, lay.tail_k, lay.tail_v,
                                      lay.tail_len, self.tail_cap, lay.kc, lay.ksz, lay.vc, lay.vsz,
                                      lay.packed_len, self.P_cap, self.cs)
        self.cs.synchronize()
        self.max_prefix += n_acc + 1

    # ------------------------------------------------------------ decoding
    def _shape_k(self, k):
        """Shape struct for a round that drafts k tokens (k <= the k buffers were sized for)."""
        if k == self.k:
            return self.sh
        if not hasattr(self, "_shapes"):
            self._shapes = {}
        if k not in self._shapes:
            s = self.sh
            self._shapes[k] = vc.shape(1, s.Hq, s.Hkv, s.d, k=k, bits=s.bits, softmax_scale=s.softmax_scale)
        return self._shapes[k]

    def generate(self, model, first_token, pos0, n_new, drafter="compressed", reference=None, rng=None,
                 k_policy=None):
        """Speculative decoding from the last prompt token's prediction
        ``first_token``; returns (tokens, accepted lengths).

        k_policy sets each round's draft length (1 <= k <= the decoder's k): None
        keeps the decoder's k; an object with next_k() / observe(n_acc, k) (a
        DraftLengthController) is asked before and told after every round; any
        other callable is called with the round index."""
        out = [int(first_token)]
        accepted = []
        pos = pos0
        rnd = 0
        while len(out) < n_new:
            if k_policy is None:
                kr = self.k
            elif hasattr(k_policy, "next_k"):
                kr = int(k_policy.next_k())
            else:
                kr = int(k_policy(rnd))
            if not 1 <= kr <= self.k:
                raise ValueError(f"draft length {kr} outside [1, {self.k}]")
            sh = self._shape_k(kr)
            t_last = out[-1]
            drafts = []
            cur = t_last
            for i in range(kr):
                lg, _, _ = model.forward(np.asarray([cur]), np.asarray([pos + i]),
                                         lambda l, q, kk, vv, _i=i: self.draft_attend(l, q, kk, vv, _i))
                if drafter == "compressed":
                    cur = int(np.argmax(lg[-1]))
                elif drafter == "wrong":
                    idx = len(out) + i
                    cur = ((reference[idx] if idx < len(reference) else 0) + 1) % self.V
                elif drafter == "perfect":
                    idx = len(out) + i
                    cur = reference[idx] if idx < len(reference) else 0
                elif drafter == "random":
                    cur = int(rng.integers(0, self.V))
                else:
                    raise ValueError(drafter)
                drafts.append(cur)
            inputs = np.asarray([t_last] + drafts)
            vlg, _, _ = model.forward(inputs, pos + np.arange(kr + 1),
                                      lambda l, q, kk, vv: self.verify_attend(l, q, kk, vv, sh=sh))
            n, nxt = self.accept(vlg, drafts)
            accepted.append(n)
            if hasattr(k_policy, "observe"):
                k_policy.observe([n], kr)
            self.commit(n, sh=sh)
            rnd += 1
            pos += n + 1
            out.extend(drafts[:n])
            out.append(nxt)
        return out[:n_new], accepted

    def greedy(self, model, first_token, pos0, n_new):
        """Plain greedy full-KV decoding through the same verify kernel (k = 0)."""
        out = [int(first_token)]
        pos = pos0
        while len(out) < n_new:
            lg, _, _ = model.forward(np.asarray([out[-1]]), np.asarray([pos]),
                                     lambda l, q, kk, vv: self.verify_attend(l, q, kk, vv, sh=self.sh0))
            self.commit(0, sh=self.sh0, append_draft=False)
            pos += 1
            out.append(int(np.argmax(lg[-1])))
        return out
