"""The lossless invariant on the oracle: draft/verify/accept == greedy full-KV.

VeriCache, Technical Summary, Experimental Results (Correctness): under greedy
decoding the output equals full-KV inference.  Checked for every compressor
(int4, int2, token drop + int4) and for drafters of any quality, plus a
planted mistake in the accept rule that must break it.
"""
import numpy as np
import pytest

import oracle.loop as loop
from oracle import tokendrop as td
from tiny_model import TinyDecoder

PROMPT_LEN = 200
N_NEW = 48


@pytest.fixture(scope="module")
def setup():
    m = TinyDecoder()
    prompt = np.random.default_rng(9).integers(0, m.vocab, PROMPT_LEN)
    ref = loop.greedy_decode(m, prompt, N_NEW, m.scale)
    return m, prompt, ref


def drop_quarter(layer, K, V, q):
    """Token dropping: score with the last 32 prompt queries, keep 25% incl. the last 32."""
    T = K.shape[1]
    qo = np.asarray(q)[-32:].transpose(1, 0, 2)[None]          # [1, Hq, 32, d]
    s = td.token_scores(qo, K[None], 1 / 8)
    idx = td.select_tokens(td.max_pool(s), T // 4 // 32 * 32, 32)
    return td.gather(K[None], idx)[0], td.gather(V[None], idx)[0]


@pytest.mark.parametrize("bits,compress", [(4, None), (2, None), (4, drop_quarter)], ids=["int4", "int2", "drop+int4"])
def test_lossless_compressed_drafter(setup, bits, compress):
    m, prompt, ref = setup
    out, acc = loop.speculative_decode(m, prompt, N_NEW, 4, bits, m.scale, compress=compress)
    assert out == ref
    assert len(acc) < N_NEW                 # drafting made progress beyond 1 token per round
    assert sum(a + 1 for a in acc) >= N_NEW


@pytest.mark.parametrize("drafter", ["wrong", "perfect", "random"])
def test_lossless_any_drafter(setup, drafter):
    m, prompt, ref = setup
    out, acc = loop.speculative_decode(m, prompt, N_NEW, 4, 4, m.scale, drafter=drafter,
                                       rng=np.random.default_rng(0), reference=ref)
    assert out == ref
    if drafter == "wrong":
        assert all(a == 0 for a in acc)
    if drafter == "perfect":
        assert all(a == 4 for a in acc[:-1])


def test_planted_accept_mistake_breaks_identity(setup, monkeypatch):
    """Accepting one token past the first mismatch must change the stream."""
    m, prompt, ref = setup
    good = loop.accept_rule

    def off_by_one(logits, draft):
        n, nxt, a = good(logits, draft)
        k = draft.shape[1]
        n2 = np.minimum(n + 1, k).astype(np.int32)
        return n2, a[np.arange(a.shape[0]), n2].astype(np.int32), a

    monkeypatch.setattr(loop, "accept_rule", off_by_one)
    out, _ = loop.speculative_decode(m, prompt, N_NEW, 4, 2, m.scale, drafter="random",
                                     rng=np.random.default_rng(0), reference=ref)
    assert out != ref
