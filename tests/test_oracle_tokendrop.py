"""Pins for the oracle's SnapKV-style token dropping.

Closed forms (identical keys give uniform causal rows), the per-row sum
identity, hand-built pooled maxima, an O(T^2) rank definition of the top-k
selection, and the identity / last-32 invariants.
"""
import numpy as np
import pytest

import synth
from oracle import tokendrop as td


def _bits(x):
    return synth.bf16_bits(np.asarray(x, np.float32))


def test_identical_keys_closed_form():
    B, Hq, Hkv, T, d, n_obs = 1, 4, 2, 100, 64, 32
    rng = np.random.default_rng(0)
    key = rng.standard_normal(d)
    K = _bits(np.broadcast_to(key, (B, Hkv, T, d)))
    q = _bits(rng.standard_normal((B, Hq, n_obs, d)))
    s = td.token_scores(q, K, 1.0)
    G = Hq // Hkv
    want = np.zeros(T)
    for i in range(n_obs):
        last = T - n_obs + i
        want[:last + 1] += 1.0 / (last + 1)
    assert np.allclose(s[0, 0], G * want, rtol=1e-12, atol=1e-12)
    assert np.allclose(s[0, 1], G * want, rtol=1e-12, atol=1e-12)


def test_row_sums_and_causality():
    rng = np.random.default_rng(1)
    B, Hq, Hkv, T, d = 2, 6, 2, 80, 64
    q = _bits(rng.standard_normal((B, Hq, 32, d)) / 8)
    K = _bits(rng.standard_normal((B, Hkv, T, d)))
    s = td.token_scores(q, K, 1.0)
    # every softmax row sums to one: the total mass per KV head is G * 32
    assert np.allclose(s.sum(-1), (Hq // Hkv) * 32, rtol=1e-12)
    # the last key is seen only by the last query of each head: s = sum_h p_h
    assert np.all(s[..., -1] > 0) and np.all(s[..., -1] < Hq // Hkv)


def test_max_pool_by_hand():
    s = np.zeros((1, 1, 20))
    s[0, 0, 0] = 5.0
    s[0, 0, 10] = 2.0
    s[0, 0, 19] = 1.0
    p = td.max_pool(s)
    want = np.zeros(20)
    want[0:4] = 5.0          # window of t=0..3 reaches t=0
    want[7:14] = 2.0         # 10-3 .. 10+3
    want[16:20] = 1.0        # 19-3 .. 19 (clipped)
    assert np.array_equal(p[0, 0], want)


def _rank_select(pooled, keep, keep_last):
    """Token t < T-keep_last is kept iff fewer than keep-keep_last candidates beat it
    (a higher score, or an equal score at a lower index)."""
    T = pooled.shape[0]
    cand = T - keep_last
    kept = []
    for t in range(cand):
        beat = sum(1 for u in range(cand) if pooled[u] > pooled[t] or (pooled[u] == pooled[t] and u < t))
        if beat < keep - keep_last:
            kept.append(t)
    return kept + list(range(cand, T))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_select_equals_rank_definition(seed):
    rng = np.random.default_rng(seed)
    T, keep = 64, 48
    pooled = rng.integers(0, 6, size=(2, 2, T)).astype(np.float64)   # many ties
    idx = td.select_tokens(pooled, keep, 32)
    for b in range(2):
        for h in range(2):
            assert idx[b, h].tolist() == _rank_select(pooled[b, h], keep, 32)


def test_select_identity_and_last_tokens():
    rng = np.random.default_rng(3)
    pooled = rng.random((1, 3, 256))
    assert np.array_equal(td.select_tokens(pooled, 256, 32)[0], np.tile(np.arange(256), (3, 1)))
    idx = td.select_tokens(pooled, 64, 32)
    assert np.all(np.diff(idx, axis=-1) > 0)
    assert np.all(idx[..., -32:] == np.arange(224, 256))


def test_gather():
    X = np.arange(2 * 3 * 10 * 4).reshape(2, 3, 10, 4)
    idx = np.array([[[1, 5], [0, 9], [2, 3]], [[4, 4], [8, 1], [7, 0]]], np.int32)
    g = td.gather(X, idx)
    for b in range(2):
        for h in range(3):
            for j in range(2):
                assert np.array_equal(g[b, h, j], X[b, h, idx[b, h, j]])
