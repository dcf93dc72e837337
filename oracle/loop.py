"""The draft -> verify -> accept loop and the lossless invariant (oracle).

VeriCache, Technical Summary, Core Algorithm: draft candidate tokens with the
compressed cache, verify them in one forward pass over the full cache, keep
them up to the first disagreement (plus the full-KV token there), and repeat
from the last kept token.  Architecture Support, long-context decoding: the
compressed cache sits in GPU memory, the full cache in CPU memory.  The
output must equal plain greedy decoding with the full cache (Experimental
Results, Correctness).

The model is anything with the small interface below (``DecoderModel``);
the tests use a tiny random-init decoder.  Attention is the only part this
oracle defines; the rest of the model is the caller's.

Draft-cache bookkeeping (the pages are silent; this library's reading):

* the draft cache of a request is a packed prefix (a multiple of 32 tokens)
  plus a bf16 tail of committed-but-unpacked tokens;
* draft step i writes the current token's approximate K/V at tail position
  tail_len + i and attends over packed + tail[0 : tail_len + i] + itself;
* after accept, the draft entries are dropped, the EXACT K/V of the n+1
  committed tokens (the verify pass's) are appended to the tail and to the
  full cache, and while the tail holds >= 32 tokens its oldest 32 are
  quantised into the packed prefix.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Protocol

import numpy as np

from . import kivi
from .accept import accept as accept_rule
from .attention import round_bf16


class DecoderModel(Protocol):
    """What the loop needs from a model (one request, all layers).

    ``forward(tokens, positions, attend)`` runs the model on new tokens and
    returns (logits [n, V], per-layer K [L][n, Hkv, d] and V likewise, as bf16
    bits).  ``attend(layer, q, k, v)`` is called once per layer with the new
    tokens' q [n, Hq, d], k/v [n, Hkv, d] (bf16 bits) and returns the
    attention output [n, Hq, d] (any float).
    """
    n_layers: int

    def forward(self, tokens, positions, attend): ...


@dataclasses.dataclass
class DraftCache:
    """One layer's compressed cache for one request (logical, unpacked form)."""
    bits: int
    kcode: np.ndarray     # uint8 [1, Hkv, P, d]
    ks: np.ndarray        # fp16 [1, Hkv, P/32, d]
    kz: np.ndarray
    vcode: np.ndarray
    vs: np.ndarray        # fp16 [1, Hkv, P, d/32]
    vz: np.ndarray
    tail_k: np.ndarray    # bf16 bits [Hkv, n_tail, d]
    tail_v: np.ndarray

    @property
    def packed_len(self) -> int:
        return self.kcode.shape[2]

    def dequant(self):
        Kh, Vh = kivi.dequantize_kv(self.kcode, self.ks, self.kz, self.vcode, self.vs, self.vz)
        return Kh[0], Vh[0]


def new_draft_cache(K, V, bits: int) -> DraftCache:
    """Compress a request's prefix K/V [Hkv, T, d]: whole 32-groups packed, rest in the tail."""
    Hkv, T, d = K.shape
    P = (T // 32) * 32
    kc, ks, kz, vc, vs, vz = kivi.quantize_kv(K[None, :, :P], V[None, :, :P], bits)
    return DraftCache(bits, kc, ks, kz, vc, vs, vz, K[:, P:].copy(), V[:, P:].copy())


def commit_to_draft_cache(dc: DraftCache, k_new, v_new):
    """Append exact K/V [Hkv, n, d] to the tail; pack whole 32-groups from its front."""
    dc.tail_k = np.concatenate([dc.tail_k, k_new], axis=1)
    dc.tail_v = np.concatenate([dc.tail_v, v_new], axis=1)
    while dc.tail_k.shape[1] >= 32:
        kc, ks, kz, vc, vs, vz = kivi.quantize_kv(dc.tail_k[None, :, :32], dc.tail_v[None, :, :32], dc.bits)
        dc.kcode = np.concatenate([dc.kcode, kc], axis=2)
        dc.ks = np.concatenate([dc.ks, ks], axis=2)
        dc.kz = np.concatenate([dc.kz, kz], axis=2)
        dc.vcode = np.concatenate([dc.vcode, vc], axis=2)
        dc.vs = np.concatenate([dc.vs, vs], axis=2)
        dc.vz = np.concatenate([dc.vz, vz], axis=2)
        dc.tail_k = dc.tail_k[:, 32:]
        dc.tail_v = dc.tail_v[:, 32:]


def committed_kv(vk, vv, n: int, draft_k=None, draft_v=None):
    """The K/V a round appends to one layer's draft cache ([Hkv, n+1, d] each).

    They are the verify pass's exact K/V of t_last, d_0 .. d_{n-1} (vk/vv
    [k+1, Hkv, d]); the draft pass's approximate K/V of the same tokens
    (draft_k/draft_v, [Hkv, d] per draft step) are discarded.  The pages
    leave the choice open (Core Algorithm: the next round "repeats from the
    last accepted token"); exact K/V keep the draft cache equal to the
    compression of the full cache.
    """
    del draft_k, draft_v
    k = np.ascontiguousarray(np.asarray(vk)[:n + 1].transpose(1, 0, 2))
    v = np.ascontiguousarray(np.asarray(vv)[:n + 1].transpose(1, 0, 2))
    return k, v


def _bf16_to_f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _attend_rows(q, Ks, Vs, limits, scale):
    """q [n,Hq,d] f64; Ks/Vs [Hkv,N,d] f64; row r sees keys 0..limits[r]-1."""
    n, Hq, d = q.shape
    Hkv = Ks.shape[0]
    G = Hq // Hkv
    out = np.empty((n, Hq, d))
    for r in range(n):
        L = limits[r]
        for h in range(Hq):
            K = Ks[h // G, :L]
            V = Vs[h // G, :L]
            logit = scale * (K @ q[r, h])
            p = np.exp(logit - logit.max())
            out[r, h] = (p @ V) / p.sum()
    return out


class FullKV:
    """Exact K/V of every committed token, per layer (the full cache)."""

    def __init__(self, n_layers):
        self.K = [None] * n_layers
        self.V = [None] * n_layers

    def append(self, layer, k, v):          # k, v [n, Hkv, d] bf16 bits
        k = np.ascontiguousarray(np.asarray(k).transpose(1, 0, 2))
        v = np.ascontiguousarray(np.asarray(v).transpose(1, 0, 2))
        if self.K[layer] is None:
            self.K[layer], self.V[layer] = k, v
        else:
            self.K[layer] = np.concatenate([self.K[layer], k], axis=1)
            self.V[layer] = np.concatenate([self.V[layer], v], axis=1)

    def length(self):
        return 0 if self.K[0] is None else self.K[0].shape[1]


def full_attention_fn(store: FullKV, scale: float, bf16_out: bool = False):
    """Attention of new tokens over the full cache + themselves (causal).

    bf16_out rounds the fp64 result to bf16 (nearest, ties to even), the
    precision in which the attention kernels hand their output back.
    """
    def attend(layer, q, k, v):
        out = _attend_full(layer, q, k, v)
        return round_bf16(out) if bf16_out else out

    def _attend_full(layer, q, k, v):
        qf = _bf16_to_f64(q)
        T = store.length()
        Ks = _bf16_to_f64(k).transpose(1, 0, 2)
        Vs = _bf16_to_f64(v).transpose(1, 0, 2)
        if T:
            Ks = np.concatenate([_bf16_to_f64(store.K[layer]), Ks], axis=1)
            Vs = np.concatenate([_bf16_to_f64(store.V[layer]), Vs], axis=1)
        n = q.shape[0]
        return _attend_rows(qf, Ks, Vs, [T + r + 1 for r in range(n)], scale)
    return attend


def greedy_decode(model: DecoderModel, prompt, n_new: int, scale: float, bf16_out: bool = False):
    """Plain greedy decoding with full-KV attention: the reference stream."""
    store = FullKV(model.n_layers)
    logits, ks, vs = model.forward(np.asarray(prompt), np.arange(len(prompt)),
                                   full_attention_fn(store, scale, bf16_out))
    for l in range(model.n_layers):
        store.append(l, ks[l], vs[l])
    out = [int(np.argmax(logits[-1]))]
    while len(out) < n_new:
        pos = store.length()
        logits, ks, vs = model.forward(np.asarray([out[-1]]), np.asarray([pos]),
                                       full_attention_fn(store, scale, bf16_out))
        for l in range(model.n_layers):
            store.append(l, ks[l], vs[l])
        out.append(int(np.argmax(logits[-1])))
    return out


def speculative_decode(model: DecoderModel, prompt, n_new: int, k: int, bits: int,
                       scale: float, drafter: str = "compressed", rng=None,
                       reference: list | None = None, compress: Callable | None = None,
                       on_commit: Callable | None = None):
    """Draft with the compressed cache, verify with the full one, accept.

    drafter: "compressed" (the method), "wrong" (every draft is wrong),
    "perfect" (drafts copied from ``reference``), "random".  ``compress``
    optionally inserts a token-dropping step before quantisation: it maps
    (layer, K [Hkv,T,d], V, prompt queries [T,Hq,d]) to the (K, V) the draft
    cache is built from.  ``on_commit(store, caches)``, if given, sees the
    full cache and every layer's draft cache after each round's commit.
    Returns (tokens, accepted lengths per round).
    """
    L = model.n_layers
    store = FullKV(L)
    prompt_q = [None] * L
    full = full_attention_fn(store, scale)

    def prefill_attend(layer, q, k, v):
        prompt_q[layer] = q
        return full(layer, q, k, v)

    logits, ks, vs = model.forward(np.asarray(prompt), np.arange(len(prompt)), prefill_attend)
    for l in range(L):
        store.append(l, ks[l], vs[l])
    caches = []
    for l in range(L):
        Kp, Vp = store.K[l], store.V[l]
        if compress is not None:
            Kp, Vp = compress(l, Kp, Vp, prompt_q[l])
        caches.append(new_draft_cache(Kp, Vp, bits))
    out = [int(np.argmax(logits[-1]))]
    accepted = []
    while len(out) < n_new:
        t_last = out[-1]
        pos0 = store.length()
        # ---- draft k tokens with the compressed cache
        drafts = []
        extra_k = [[] for _ in range(L)]
        extra_v = [[] for _ in range(L)]
        cur = t_last
        for i in range(k):
            def draft_attend(layer, q, kk, vv, _i=i):
                dc = caches[layer]
                Kh, Vh = dc.dequant()
                parts_k = [Kh.astype(np.float64), _bf16_to_f64(dc.tail_k)]
                parts_v = [Vh.astype(np.float64), _bf16_to_f64(dc.tail_v)]
                for e in range(_i):
                    parts_k.append(_bf16_to_f64(extra_k[layer][e])[:, None])
                    parts_v.append(_bf16_to_f64(extra_v[layer][e])[:, None])
                parts_k.append(_bf16_to_f64(kk).transpose(1, 0, 2))
                parts_v.append(_bf16_to_f64(vv).transpose(1, 0, 2))
                Ks = np.concatenate(parts_k, axis=1)
                Vs = np.concatenate(parts_v, axis=1)
                extra_k[layer].append(np.asarray(kk)[0])
                extra_v[layer].append(np.asarray(vv)[0])
                return _attend_rows(_bf16_to_f64(q), Ks, Vs, [Ks.shape[1]], scale)
            lg, _, _ = model.forward(np.asarray([cur]), np.asarray([pos0 + i]), draft_attend)
            if drafter == "compressed":
                cur = int(np.argmax(lg[-1]))
            elif drafter == "wrong":
                # never the reference token at this position
                ref = reference[len(out) + i] if len(out) + i < len(reference) else 0
                cur = (ref + 1) % lg.shape[-1]
            elif drafter == "perfect":
                cur = reference[len(out) + i] if len(out) + i < len(reference) else 0
            elif drafter == "random":
                cur = int(rng.integers(0, lg.shape[-1]))
            else:
                raise ValueError(drafter)
            drafts.append(cur)
        # ---- verify: one forward pass over [t_last, d_0 .. d_{k-1}] with the full cache
        inputs = np.asarray([t_last] + drafts)
        vlogits, vks, vvs = model.forward(inputs, pos0 + np.arange(k + 1), full_attention_fn(store, scale))
        n_acc, nxt, _ = accept_rule(vlogits[None].astype(np.float32), np.asarray(drafts, np.int32)[None])
        n = int(n_acc[0])
        accepted.append(n)
        # ---- commit the exact K/V of t_last, d_0 .. d_{n-1}
        for l in range(L):
            store.append(l, vks[l][:n + 1], vvs[l][:n + 1])
            kk, vv = committed_kv(vks[l], vvs[l], n, extra_k[l], extra_v[l])
            commit_to_draft_cache(caches[l], kk, vv)
        if on_commit is not None:
            on_commit(store, caches)
        out.extend(drafts[:n])
        out.append(int(nxt[0]))
    return out[:n_new], accepted
