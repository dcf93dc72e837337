"""A tiny random-init decoder for the lossless-invariant tests.

Two layers, Hq=4 query heads over Hkv=1 KV head of dim 64 (d_model 256),
vocab 1024, RMSNorm, RoPE (theta 1e4) applied before caching, a SiLU-gated
MLP of width 512, weights N(0, 1/fan_in) and the unembedding scaled by 4 so
that logit margins are wide.  Everything except attention runs here in fp32
numpy; attention is whatever callable the caller passes, so the same model
runs on the oracle or on the CUDA kernels.

q, k and v are rounded to bf16 before they reach attention (the caches hold
bf16); the attention output comes back as floats and the rest stays fp32.
"""
from __future__ import annotations

import numpy as np

import synth


class TinyDecoder:
    def __init__(self, seed: int = 7, n_layers: int = 2, Hq: int = 4, Hkv: int = 1,
                 d: int = 64, vocab: int = 1024, d_ff: int = 512, theta: float = 1e4):
        rng = np.random.Generator(np.random.PCG64(seed))
        self.n_layers, self.Hq, self.Hkv, self.d = n_layers, Hq, Hkv, d
        self.D = Hq * d
        self.vocab = vocab
        self.theta = theta
        D = self.D

        def w(fan_in, *shape):
            return (rng.standard_normal(shape, dtype=np.float32) / np.float32(np.sqrt(fan_in))).astype(np.float32)

        self.embed = rng.standard_normal((vocab, D), dtype=np.float32)
        self.layers = []
        for _ in range(n_layers):
            self.layers.append(dict(
                wq=w(D, D, Hq * d), wk=w(D, D, Hkv * d), wv=w(D, D, Hkv * d),
                wo=w(Hq * d, Hq * d, D), w1=w(D, D, d_ff), w3=w(D, D, d_ff), w2=w(d_ff, d_ff, D)))
        self.unembed = w(D, D, vocab) * np.float32(4.0)
        self.scale = 1.0 / np.sqrt(d)

    @staticmethod
    def _rms(x):
        return (x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + np.float32(1e-6))).astype(np.float32)

    def _rope(self, x, pos):
        # x [n, H, d]; rotate-half convention
        d = x.shape[-1]
        half = d // 2
        inv = (1.0 / (self.theta ** (np.arange(half, dtype=np.float64) * 2.0 / d)))
        ang = np.asarray(pos, np.float64)[:, None] * inv[None, :]
        c = np.cos(ang).astype(np.float32)[:, None, :]
        s = np.sin(ang).astype(np.float32)[:, None, :]
        x1, x2 = x[..., :half], x[..., half:]
        return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1).astype(np.float32)

    def forward(self, tokens, positions, attend):
        """tokens [n] -> (logits [n, V] fp32, K list [L][n,Hkv,d] bf16 bits, V list)."""
        tokens = np.asarray(tokens)
        n = tokens.shape[0]
        x = self.embed[tokens].astype(np.float32)
        ks, vs = [], []
        for li, p in enumerate(self.layers):
            h = self._rms(x)
            q = (h @ p["wq"]).reshape(n, self.Hq, self.d)
            k = (h @ p["wk"]).reshape(n, self.Hkv, self.d)
            v = (h @ p["wv"]).reshape(n, self.Hkv, self.d)
            q = self._rope(q, positions)
            k = self._rope(k, positions)
            qb, kb, vb = synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v)
            ks.append(kb)
            vs.append(vb)
            a = np.asarray(attend(li, qb, kb, vb), dtype=np.float32).reshape(n, self.Hq * self.d)
            x = (x + a @ p["wo"]).astype(np.float32)
            h = self._rms(x)
            g = h @ p["w1"]
            u = h @ p["w3"]
            x = (x + ((g / (1.0 + np.exp(-g))) * u).astype(np.float32) @ p["w2"]).astype(np.float32)
        logits = (self._rms(x) @ self.unembed).astype(np.float32)
        return logits, ks, vs
