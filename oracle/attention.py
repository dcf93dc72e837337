"""Draft and verify attention (oracle), fp64.

* Draft: "The model generates a sequence of candidate tokens using the
  compressed KV cache" (VeriCache, Technical Summary, Core Algorithm,
  Drafting).  One query token per request per step, over the dequantised
  packed prefix followed by the bf16 tail of not-yet-packed tokens and the
  current token's own K/V.
* Verify: "a single forward pass using the full KV cache to verify the
  drafted tokens in parallel" (same section, Verification).  Row j of the
  k+1 verify rows attends to the T prefix tokens plus new tokens 0..j.

GQA grouping: query head h uses KV head h // G (contiguous groups).
``scale`` multiplies q.k before the softmax.  Everything is computed in fp64;
outputs are returned in fp64 (``round_bf16`` rounds to the bf16 grid).
"""
from __future__ import annotations

import numpy as np

from .kivi import unpack_dequant


def _bf16_to_f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (8 significant bits, ties to even), as fp64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                     # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def softmax_attend(q, K, V, scale: float):
    """o = softmax(scale * q.K^T) V for one query vector (fp64).

    q [d], K [n, d], V [n, d] -> o [d].  Subtracting the max is exact
    algebra (it cancels between numerator and denominator).
    """
    logit = scale * (K @ q)
    p = np.exp(logit - logit.max())
    return (p @ V) / p.sum()


def decode_attention(q, K, V, scale: float):
    """Decode attention over a full-precision KV (fp64 result).

    q [B, Hq, d]; K, V [B, Hkv, T, d] (any float dtype).  Returns [B, Hq, d].
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.empty((B, Hq, d))
    for b in range(B):
        for h in range(Hq):
            out[b, h] = softmax_attend(q[b, h], K[b, h // G], V[b, h // G], scale)
    return out


def draft_attention(q, kc, ksz, vc, vsz, packed_len, tail_k, tail_v, tail_len,
                    bits: int, scale: float, k_cur=None, v_cur=None, step: int = 0):
    """Draft decode attention over the compressed cache (fp64 result).

    q [B,Hq,d] bf16 bits; packed cache in the library layout; packed_len [B];
    tail_k/tail_v [B,Hkv,R,d] bf16 bits; tail_len [B].
    Request b attends to: dequant(packed tokens 0..packed_len[b]-1), then tail
    entries 0..tail_len[b]+step-1, then, if given, the current token's
    k_cur/v_cur [B,Hkv,d] (its own K/V), in that order.
    """
    qf = _bf16_to_f64(q)
    B, Hq, d = qf.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    Kh, Vh = unpack_dequant(kc, ksz, vc, vsz, bits, d)
    tk = _bf16_to_f64(tail_k)
    tv = _bf16_to_f64(tail_v)
    out = np.empty((B, Hq, d))
    for b in range(B):
        P = int(packed_len[b])
        R = int(tail_len[b]) + step
        for kvh in range(Hkv):
            Ks = [Kh[b, kvh, :P].astype(np.float64), tk[b, kvh, :R]]
            Vs = [Vh[b, kvh, :P].astype(np.float64), tv[b, kvh, :R]]
            if k_cur is not None:
                Ks.append(_bf16_to_f64(k_cur)[b, kvh][None])
                Vs.append(_bf16_to_f64(v_cur)[b, kvh][None])
            Kall = np.concatenate(Ks)
            Vall = np.concatenate(Vs)
            for g in range(G):
                h = kvh * G + g
                out[b, h] = softmax_attend(qf[b, h], Kall, Vall, scale)
    return out


def verify_attention(q, K, V, k_new, v_new, prefix_len, scale: float):
    """Verify attention for the k+1 rows of each request (fp64 result).

    q [B,k+1,Hq,d]; K,V [B,Hkv,Tmax,d] full prefix (bf16 bits); prefix_len [B]
    tokens of it are valid; k_new/v_new [B,k+1,Hkv,d] exact K/V of the verify
    inputs.  Row j sees prefix tokens 0..prefix_len[b]-1 and new tokens 0..j.
    Returns [B,k+1,Hq,d].
    """
    qf = _bf16_to_f64(q)
    Kf = _bf16_to_f64(K)
    Vf = _bf16_to_f64(V)
    kn = _bf16_to_f64(k_new)
    vn = _bf16_to_f64(v_new)
    B, R, Hq, d = qf.shape
    Hkv = Kf.shape[1]
    G = Hq // Hkv
    out = np.empty((B, R, Hq, d))
    for b in range(B):
        T = int(prefix_len[b])
        for kvh in range(Hkv):
            for j in range(R):
                Kall = np.concatenate([Kf[b, kvh, :T], kn[b, :j + 1, kvh]])
                Vall = np.concatenate([Vf[b, kvh, :T], vn[b, :j + 1, kvh]])
                for g in range(G):
                    h = kvh * G + g
                    out[b, j, h] = softmax_attend(qf[b, j, h], Kall, Vall, scale)
    return out
