"""Seeded synthetic inputs for the VeriCache draft -> verify -> accept hot path.

This module only draws random numbers and stores them in the layouts the
library and the oracle both read.  It holds none of the method's arithmetic:
no quantisation, no attention, no argmax.  Both the CUDA path (through the
tests and the benchmark) and the CPU oracle take their inputs from here.

Every tensor is drawn from ``numpy.random.Generator(PCG64)`` seeded by a
``SeedSequence`` of (workload seed, tensor id, slice indices), so any single
(request, head) slice of a large tensor can be regenerated on its own without
drawing the rest.  bf16 tensors are returned as ``uint16`` bit patterns,
rounded to nearest-even from the fp32 draw.

The shapes and value distributions stand in for the workloads the VeriCache
page evaluates on (Mistral-24B, Qwen-32B and Llama-70B serving code, tool and
math tasks; gist.science/paper/2605.17613, Technical Summary, Experimental
Results): only attention-layer shapes are used, since neither the models'
weights nor the evaluation suites are available.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "get", "bf16_bits", "bf16_to_f32",
    "draft_q", "verify_q", "kv_slice", "kv", "kv_new", "logits_and_drafts",
    "q_obs", "outlier_channels", "accept_lengths",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int          # requests in the batch (per group for the staggered mix)
    Hq: int         # query heads
    Hkv: int        # KV heads
    d: int          # head dim
    T: int          # context tokens held in the full KV at the start
    k: int          # draft length per round
    bits: int       # KIVI code width for the draft cache
    V: int          # vocabulary size of the logits the accept step reads
    C: int          # tokens per host->device chunk of the full KV
    layers: int = 1
    n_outlier: int = 4
    accept: str = "geom"     # "uniform" (Tiny) or "geom"
    p_geom: float = 0.1
    keep_frac: float = 1.0   # token dropping keeps this fraction (1.0 = none)
    groups: int = 1          # staggered request groups
    rounds: int = 1          # rounds the staggered schedule runs

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def T_keep(self) -> int:
        return int(round(self.T * self.keep_frac))


# Shapes and distributions of the five workloads.  Seeds are 1000 + index.
WORKLOADS = {
    "tiny": Workload("tiny", 1000, B=1, Hq=4, Hkv=1, d=64, T=512, k=4, bits=4,
                     V=1024, C=128, n_outlier=2, accept="uniform"),
    "mistral": Workload("mistral", 1001, B=8, Hq=32, Hkv=8, d=128, T=32768, k=16,
                        bits=2, V=32768, C=4096, p_geom=0.1),
    "qwen": Workload("qwen", 1002, B=16, Hq=40, Hkv=8, d=128, T=65536, k=32,
                     bits=4, V=152064, C=4096, p_geom=0.05, keep_frac=0.25),
    "llama": Workload("llama", 1003, B=4, Hq=64, Hkv=8, d=128, T=131072, k=32,
                      bits=2, V=128256, C=4096, layers=8, p_geom=0.04),
    "stagger": Workload("stagger", 1004, B=32, Hq=32, Hkv=8, d=128, T=32768, k=24,
                        bits=2, V=128256, C=4096, p_geom=0.06, groups=2, rounds=50),
}


def get(name: str, **overrides) -> Workload:
    """A workload by name, optionally with fields replaced (smaller cases)."""
    return dataclasses.replace(WORKLOADS[name], **overrides)


# ---------------------------------------------------------------- bf16 bits

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------- streams

_TENSOR_IDS = {"q_draft": 1, "q_verify": 2, "K": 3, "V": 4, "k_new": 5,
               "v_new": 6, "logits": 7, "draft": 8, "accept": 9, "q_obs": 10,
               "outliers": 11, "bonus": 12, "k_cur": 13, "v_cur": 14}


def _rng(w: Workload, tensor: str, *idx: int) -> np.random.Generator:
    ss = np.random.SeedSequence([w.seed, _TENSOR_IDS[tensor], *[int(i) for i in idx]])
    return np.random.Generator(np.random.PCG64(ss))


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def outlier_channels(w: Workload, layer: int, h: int) -> np.ndarray:
    """The key channels of KV head ``h`` that are scaled by 10."""
    rng = _rng(w, "outliers", layer, h)
    return np.sort(rng.choice(w.d, size=w.n_outlier, replace=False))


# ---------------------------------------------------------------- tensors

def draft_q(w: Workload, rnd: int, step: int, layer: int = 0, group: int = 0) -> np.ndarray:
    """Query of draft step ``step`` of round ``rnd``: bf16 bits [B, Hq, d], N(0,1)/sqrt(d)."""
    rng = _rng(w, "q_draft", group, layer, rnd, step)
    return bf16_bits(_normal(rng, (w.B, w.Hq, w.d)) / np.float32(math.sqrt(w.d)))


def draft_kv_cur(w: Workload, rnd: int, step: int, layer: int = 0, group: int = 0):
    """K/V of the token a draft step feeds in: bf16 bits [B, Hkv, d] each."""
    rk = _rng(w, "k_cur", group, layer, rnd, step)
    rv = _rng(w, "v_cur", group, layer, rnd, step)
    return (bf16_bits(_normal(rk, (w.B, w.Hkv, w.d))),
            bf16_bits(_normal(rv, (w.B, w.Hkv, w.d))))


def verify_q(w: Workload, rnd: int, layer: int = 0, group: int = 0) -> np.ndarray:
    """Queries of the k+1 verify rows: bf16 bits [B, k+1, Hq, d]."""
    rng = _rng(w, "q_verify", group, layer, rnd)
    return bf16_bits(_normal(rng, (w.B, w.k + 1, w.Hq, w.d)) / np.float32(math.sqrt(w.d)))


def kv_new(w: Workload, rnd: int, layer: int = 0, group: int = 0):
    """Exact K/V of the k+1 verify inputs: bf16 bits [B, k+1, Hkv, d] each."""
    rk = _rng(w, "k_new", group, layer, rnd)
    rv = _rng(w, "v_new", group, layer, rnd)
    return (bf16_bits(_normal(rk, (w.B, w.k + 1, w.Hkv, w.d))),
            bf16_bits(_normal(rv, (w.B, w.k + 1, w.Hkv, w.d))))


def kv_slice(w: Workload, b: int, h: int, layer: int = 0, group: int = 0, T: int | None = None):
    """Prefix K and V of request ``b``, KV head ``h``: bf16 bits [T, d] each.

    K ~ N(0,1) with ``n_outlier`` channels scaled by 10; V ~ N(0,1).
    """
    T = w.T if T is None else T
    k = _normal(_rng(w, "K", group, layer, b, h), (T, w.d))
    k[:, outlier_channels(w, layer, h)] *= np.float32(10.0)
    v = _normal(_rng(w, "V", group, layer, b, h), (T, w.d))
    return bf16_bits(k), bf16_bits(v)


def kv(w: Workload, layer: int = 0, group: int = 0, T: int | None = None, threads: int = 8):
    """Full prefix K and V: bf16 bits [B, Hkv, T, d] each."""
    T = w.T if T is None else T
    K = np.empty((w.B, w.Hkv, T, w.d), np.uint16)
    Vv = np.empty_like(K)

    def fill(bh):
        b, h = bh
        K[b, h], Vv[b, h] = kv_slice(w, b, h, layer, group, T)

    jobs = [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    if threads > 1 and len(jobs) > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, jobs))
    else:
        for j in jobs:
            fill(j)
    return K, Vv


def q_obs(w: Workload, n_obs: int = 32, group: int = 0) -> np.ndarray:
    """Queries of the last ``n_obs`` prompt tokens: bf16 bits [B, Hq, n_obs, d]."""
    rng = _rng(w, "q_obs", group)
    return bf16_bits(_normal(rng, (w.B, w.Hq, n_obs, w.d)) / np.float32(math.sqrt(w.d)))


def accept_lengths(w: Workload, rnd: int, group: int = 0) -> np.ndarray:
    """Intended accepted length per request (int64 [B]).

    Tiny: uniform on {0..k}.  Others: min(Geom0(p), k) with P(n) = (1-p)^n p.
    """
    rng = _rng(w, "accept", group, rnd)
    if w.accept == "uniform":
        return rng.integers(0, w.k + 1, size=w.B)
    return np.minimum(rng.geometric(w.p_geom, size=w.B) - 1, w.k)


def logits_and_drafts(w: Workload, rnd: int, group: int = 0):
    """Synthetic verify logits fp32 [B, k+1, V] and draft tokens int32 [B, k].

    Logits ~ N(0,1).  For the intended accepted length L of a request, rows
    i < L get +8 at the draft token, so the full-KV prediction agrees with the
    draft there; if L < k, row L gets +8 at a token other than the draft, so
    the drafts disagree from L on.  The accept step itself (an argmax over the
    rows) decides the accepted length, not this generator.
    """
    L = accept_lengths(w, rnd, group)
    rl = _rng(w, "logits", group, rnd)
    logits = _normal(rl, (w.B, w.k + 1, w.V))
    rd = _rng(w, "draft", group, rnd)
    drafts = rd.integers(0, w.V, size=(w.B, w.k)).astype(np.int32)
    rb = _rng(w, "bonus", group, rnd)
    other = rb.integers(1, max(w.V, 2), size=w.B)
    for b in range(w.B):
        for i in range(int(L[b])):
            logits[b, i, drafts[b, i]] += np.float32(8.0)
        if L[b] < w.k and w.V > 1:
            tok = (int(drafts[b, L[b]]) + int(other[b])) % w.V
            logits[b, L[b], tok] += np.float32(8.0)
    return logits, drafts, L
