"""SnapKV-style token dropping (oracle).

VeriCache's compressor interface takes token-dropping methods too and names
SnapKV among them (VeriCache, Technical Summary, Architecture Support).  The
recipe this library implements, for each request and KV head:

1. score s[t] = sum, over the G query heads sharing the KV head and over the
   last n_obs = 32 prompt queries i, of the post-softmax attention weight that
   query i gives key t.  Query i sits at absolute position T - n_obs + i and
   sees keys 0 .. T - n_obs + i (causal).  Logits are scale * q.k; all in fp64.
2. pooled[t] = max of s over the window t-3 .. t+3 (7 wide, stride 1, the
   window clipped at both ends).
3. keep = the last n_obs tokens, plus the (keep_total - n_obs) tokens of
   0 .. T - n_obs - 1 with the largest pooled score (ties -> lower index);
   indices returned in ascending order.
4. gather the kept tokens' K and V; they are then quantised (4-bit here).
"""
from __future__ import annotations

import numpy as np


def _bf16_to_f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def token_scores(q_obs, K, scale: float) -> np.ndarray:
    """q_obs [B,Hq,n_obs,d], K [B,Hkv,T,d] (bf16 bits) -> s fp64 [B,Hkv,T]."""
    q = _bf16_to_f64(q_obs)
    Kf = _bf16_to_f64(K)
    B, Hq, n_obs, d = q.shape
    Hkv, T = Kf.shape[1], Kf.shape[2]
    G = Hq // Hkv
    s = np.zeros((B, Hkv, T))
    for b in range(B):
        for kvh in range(Hkv):
            for g in range(G):
                h = kvh * G + g
                logits = scale * (q[b, h] @ Kf[b, kvh].T)          # [n_obs, T]
                for i in range(n_obs):
                    last = T - n_obs + i                              # inclusive
                    row = logits[i, :last + 1]
                    p = np.exp(row - row.max())
                    s[b, kvh, :last + 1] += p / p.sum()
    return s


def max_pool(s: np.ndarray, width: int = 7) -> np.ndarray:
    """Same-length max-pool along the last axis, window clipped at the ends."""
    r = width // 2
    T = s.shape[-1]
    out = np.empty_like(s)
    for t in range(T):
        out[..., t] = s[..., max(0, t - r):min(T, t + r + 1)].max(axis=-1)
    return out


def select_tokens(pooled: np.ndarray, keep: int, keep_last: int = 32) -> np.ndarray:
    """pooled [B,Hkv,T] -> kept indices int32 [B,Hkv,keep], ascending."""
    B, H, T = pooled.shape
    assert keep_last <= keep <= T
    out = np.empty((B, H, keep), np.int32)
    n_top = keep - keep_last
    cand = T - keep_last
    for b in range(B):
        for h in range(H):
            sc = pooled[b, h, :cand]
            # stable sort on the negated score: equal scores keep index order
            order = np.argsort(-sc, kind="stable")[:n_top]
            idx = np.concatenate([order, np.arange(cand, T)])
            out[b, h] = np.sort(idx)
    return out


def gather(X, idx):
    """X [B,Hkv,T,d], idx [B,Hkv,n] -> X[b,h,idx[b,h]] [B,Hkv,n,d]."""
    return np.take_along_axis(X, idx[..., None].astype(np.int64), axis=2)
