"""Pins of the oracle's draft-cache bookkeeping (new_draft_cache, commit_to_draft_cache).

VeriCache, Technical Summary, Core Algorithm: drafting reads the compressed
cache; after verification the kept tokens are committed and the next round
"repeats from the last accepted token".  The pages fix no bookkeeping; the
reading this library takes is a definition, checked here against itself
being computed some other way:

  after any sequence of commits, a request's draft cache is the KIVI-style
  quantisation of the first floor(N/32)*32 tokens of the exact committed
  sequence (N tokens so far), and its bf16 tail is the remaining tokens,
  bit for bit; the committed K/V are the verify pass's exact ones.

The lossless invariant cannot see a mistake here (it holds whatever the draft
cache holds), so these tests check the cache itself, plus planted mistakes
(packing the newest 32 tail tokens, committing the draft pass's K/V) that
must fail the same checks.
"""
import numpy as np
import pytest

import oracle.loop as loop
from oracle import kivi
from tiny_model import TinyDecoder


def bf16(x):
    x = np.asarray(x, np.float32)
    b = x.view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def defined_cache(K, V, bits):
    """The definition: quantise the first floor(N/32)*32 tokens, keep the rest exact."""
    N = K.shape[1]
    P = N // 32 * 32
    return kivi.quantize_kv(K[None, :, :P], V[None, :, :P], bits), K[:, P:], V[:, P:]


def mismatches(dc, K, V):
    """Fields of draft cache dc that differ from the definition applied to K, V ([Hkv, N, d])."""
    (kc, ks, kz, vc, vs, vz), tk, tv = defined_cache(K, V, dc.bits)
    bad = []
    for name, got, want in (("kcode", dc.kcode, kc), ("ks", dc.ks, ks), ("kz", dc.kz, kz),
                            ("vcode", dc.vcode, vc), ("vs", dc.vs, vs), ("vz", dc.vz, vz),
                            ("tail_k", dc.tail_k, tk), ("tail_v", dc.tail_v, tv)):
        if got.shape != want.shape or got.dtype != want.dtype or not np.array_equal(got, want):
            bad.append(name)
    return bad


def commit_newest(dc, k_new, v_new):
    """A plausible mistake: pack the NEWEST 32 tail tokens instead of the oldest."""
    dc.tail_k = np.concatenate([dc.tail_k, k_new], axis=1)
    dc.tail_v = np.concatenate([dc.tail_v, v_new], axis=1)
    while dc.tail_k.shape[1] >= 32:
        kc, ks, kz, vc, vs, vz = kivi.quantize_kv(dc.tail_k[None, :, -32:], dc.tail_v[None, :, -32:], dc.bits)
        dc.kcode = np.concatenate([dc.kcode, kc], axis=2)
        dc.ks = np.concatenate([dc.ks, ks], axis=2)
        dc.kz = np.concatenate([dc.kz, kz], axis=2)
        dc.vcode = np.concatenate([dc.vcode, vc], axis=2)
        dc.vs = np.concatenate([dc.vs, vs], axis=2)
        dc.vz = np.concatenate([dc.vz, vz], axis=2)
        dc.tail_k = dc.tail_k[:, :-32]
        dc.tail_v = dc.tail_v[:, :-32]


def run_commits(commit, K, V, T0, sizes, bits):
    """Build from the first T0 tokens, commit the given run lengths; yield (cache, N) after each."""
    dc = loop.new_draft_cache(K[:, :T0], V[:, :T0], bits)
    yield dc, T0
    n = T0
    for s in sizes:
        commit(dc, K[:, n:n + s], V[:, n:n + s])
        n += s
        yield dc, n


def random_kv(rng, Hkv, N, d):
    K = bf16(rng.standard_normal((Hkv, N, d)).astype(np.float32) * np.float32(3.0))
    V = bf16(rng.standard_normal((Hkv, N, d)).astype(np.float32))
    return K, V


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("T0", [0, 5, 31, 32, 61, 96])
def test_commits_match_the_definition(bits, T0):
    rng = np.random.default_rng(100 + bits * 7 + T0)
    sizes = [1, 5, 33, 2, 31, 32, 17, 65, 3, 1]       # crosses group boundaries by 0, 1, many
    K, V = random_kv(rng, 2, T0 + sum(sizes), 64)
    for dc, n in run_commits(loop.commit_to_draft_cache, K, V, T0, sizes, bits):
        assert mismatches(dc, K[:, :n], V[:, :n]) == [], f"after {n} tokens"
        assert dc.packed_len == n // 32 * 32 and dc.tail_k.shape[1] == n % 32


def test_hand_worked_boundary_commit():
    """A tail of 30 plus a 5-token commit packs tokens 0..31 and leaves 32, 33, 34.

    Key channel c of token t holds t, value channel c of token t holds t, so
    (4-bit codes) the packed key group has zero fp16(0) = 0 in every channel
    and scale fp16(31/15) = 1058 * 2^-9 = 2.06640625, key codes
    rint(t / 2.06640625) (token 16 -> rint(7.743) = 8, token 31 -> 15); every
    value group is constant, so its scale is 0, its codes are 0 and its zero
    is t: the packed zeros read 0, 1, ..., 31.  The tail holds 32, 33, 34.
    """
    t = np.arange(35, dtype=np.float32)
    K = bf16(np.repeat(t[None, :, None], 32, axis=2))      # [1, 35, 32]
    V = bf16(np.repeat(t[None, :, None], 32, axis=2))
    dc = loop.new_draft_cache(K[:, :30], V[:, :30], 4)
    assert dc.packed_len == 0 and dc.tail_k.shape[1] == 30
    loop.commit_to_draft_cache(dc, K[:, 30:35], V[:, 30:35])
    assert dc.packed_len == 32 and dc.tail_k.shape[1] == 3
    assert np.all(dc.kz == 0.0) and np.all(dc.ks == np.float16(2.06640625))
    assert dc.kcode[0, 0, 0, 0] == 0 and dc.kcode[0, 0, 16, 5] == 8 and dc.kcode[0, 0, 31, 31] == 15
    assert np.array_equal(dc.vz[0, 0, :, 0].astype(np.float32), np.arange(32, dtype=np.float32))
    assert np.all(dc.vs == 0) and np.all(dc.vcode == 0)
    assert np.array_equal(dc.tail_k[0, :, 0], bf16(np.array([32.0, 33.0, 34.0], np.float32)))
    assert np.array_equal(dc.tail_v[0, :, 7], bf16(np.array([32.0, 33.0, 34.0], np.float32)))


def test_planted_newest_pack_is_caught():
    """Packing the newest 32 tail tokens must fail the definition check (and the hand case)."""
    rng = np.random.default_rng(5)
    K, V = random_kv(rng, 1, 30 + 5, 32)
    caught = [mismatches(dc, K[:, :n], V[:, :n]) for dc, n in run_commits(commit_newest, K, V, 30, [5], 4)]
    assert caught[0] == [] and caught[1] != []


@pytest.fixture(scope="module")
def tiny():
    m = TinyDecoder()
    prompt = np.random.default_rng(9).integers(0, m.vocab, 200)
    return m, prompt


@pytest.mark.parametrize("bits", [4, 2])
def test_loop_draft_cache_is_the_compressed_full_cache(tiny, bits):
    """In the running loop, after every round's commit, each layer's draft cache
    equals the definition applied to the exact full cache (prompt + commits)."""
    m, prompt = tiny
    rounds = []

    def check(store, caches):
        for l, dc in enumerate(caches):
            assert mismatches(dc, store.K[l], store.V[l]) == [], f"round {len(rounds)}, layer {l}"
        rounds.append(store.length())

    loop.speculative_decode(m, prompt, 40, 4, bits, m.scale, on_commit=check)
    assert len(rounds) >= 8 and rounds[-1] > 232       # several rounds, some crossing a group boundary


def test_planted_draft_time_commit_is_caught(tiny, monkeypatch):
    """Committing the draft pass's approximate K/V (the tokens are the same, the
    values are not, from layer 1 on) must fail the same check."""
    m, prompt = tiny
    exact = loop.committed_kv

    def draft_time_kv(vk, vv, n, draft_k, draft_v):
        k, v = exact(vk, vv, n)
        m_ = min(n + 1, len(draft_k))
        k[:, :m_] = np.stack(draft_k[:m_], axis=1)
        v[:, :m_] = np.stack(draft_v[:m_], axis=1)
        return k, v

    monkeypatch.setattr(loop, "committed_kv", draft_time_kv)
    failures = []

    def check(store, caches):
        failures.extend(mismatches(dc, store.K[l], store.V[l]) != [] for l, dc in enumerate(caches))

    out, _ = loop.speculative_decode(m, prompt, 40, 4, 4, m.scale, on_commit=check)
    assert any(failures)
    # the output itself stays lossless: only the draft cache is wrong, which is why
    # the identity test cannot see this mistake
    assert out == loop.greedy_decode(m, prompt, 40, m.scale)
