"""The draft launch's stream-K partition, computed on the host (no GPU): it
covers every packed group exactly once, in order; a slice meets no more stream
CTAs than the workspace's partial slots hold; the slot count does not depend
on max_packed; and the ranges are balanced by cost, not by groups: a CTA whose
range crosses a slice boundary takes fewer groups than one that does not."""
import bisect

import pytest


@pytest.fixture(scope="module")
def vc():
    from verify_compressed_kv_gb300 import _lib
    return _lib


SHAPES = [
    # name, B, Hq, Hkv, d, bits, max_packed, slots
    ("llama", 4, 64, 8, 128, 2, 131072, 152),
    ("llama_grown", 4, 64, 8, 128, 2, 134816, 152),
    ("mistral", 8, 32, 8, 128, 2, 32768, 152),
    ("qwen_kept", 16, 40, 8, 128, 4, 16384, 152),
    ("stagger", 32, 32, 8, 128, 2, 32768, 152),
    ("tiny", 1, 2, 2, 64, 2, 640, 152),
    ("int8_odd", 3, 5, 5, 64, 8, 96, 7),
    ("one_slot", 2, 4, 2, 128, 2, 1024, 1),
    ("many_slices", 64, 64, 8, 128, 2, 2048, 152),
]


def _slices_of(lo, n, NG, nbh):
    """(first, last) stream CTA of every slice: the CTAs holding its first and last group."""
    out = []
    for bh in range(nbh):
        first = bisect.bisect_right(lo[:n], bh * NG) - 1
        last = bisect.bisect_right(lo[:n], bh * NG + NG - 1) - 1
        out.append((first, last))
    return out


@pytest.mark.parametrize("name,B,Hq,Hkv,d,bits,P,slots", SHAPES, ids=[s[0] for s in SHAPES])
def test_partition_covers_every_group_once(vc, name, B, Hq, Hkv, d, bits, P, slots):
    s = vc.shape(B, Hq, Hkv, d, bits=bits)
    n, lo, max_parts = vc.vc_draft_attn_partition(s, P, slots)
    NG, nbh = P // 32, B * Hkv
    total = nbh * NG
    assert 1 <= n <= min(slots, 512, max(1, total // 11))
    assert len(lo) == n + 1 and lo[0] == 0 and lo[n] == total
    assert all(a <= b for a, b in zip(lo, lo[1:]))
    # ranges are non-empty until the groups run out (then every later CTA is empty)
    sizes = [b - a for a, b in zip(lo, lo[1:])]
    first_empty = next((c for c, z in enumerate(sizes) if z == 0), n)
    assert all(z == 0 for z in sizes[first_empty:])
    # every slice meets at most max_parts - 1 stream CTAs (plus its tail's slot)
    for first, last in _slices_of(lo, n, NG, nbh):
        assert 0 <= first <= last < n
        assert last - first + 2 <= max_parts


@pytest.mark.parametrize("name,B,Hq,Hkv,d,bits,P,slots", SHAPES, ids=[s[0] for s in SHAPES])
def test_partial_slots_do_not_depend_on_max_packed(vc, name, B, Hq, Hkv, d, bits, P, slots):
    """The workspace holds max_parts slots a slice: sized once for a cache's
    capacity, it must serve every smaller max_packed the rounds pass."""
    s = vc.shape(B, Hq, Hkv, d, bits=bits)
    parts = {vc.vc_draft_attn_partition(s, mp, slots)[2] for mp in sorted({32, 320, P // 2 // 32 * 32, P})}
    assert len(parts) == 1, parts


@pytest.mark.parametrize("name", ["llama", "mistral", "stagger"])
def test_ranges_balanced_by_cost(vc, name):
    """A head switch inside a range costs a flush and a ring refill: the more
    slice boundaries a CTA's range crosses, the fewer groups it takes.  The
    typical range of each class (its median: the class also holds CTAs that
    run a tail pass, and the last range, the remainder) shrinks with every
    boundary crossed, and the typical range is the class's largest but for
    the charge of one tail pass."""
    _, B, Hq, Hkv, d, bits, P, slots = next(x for x in SHAPES if x[0] == name)
    s = vc.shape(B, Hq, Hkv, d, bits=bits)
    n, lo, _ = vc.vc_draft_attn_partition(s, P, slots)
    NG = P // 32
    by_cross = {}
    for c in range(n):
        a, b = lo[c], lo[c + 1]
        by_cross.setdefault((b - 1) // NG - a // NG, []).append(b - a)
    assert len(by_cross) >= 2, by_cross.keys()
    typical = {k: sorted(v)[len(v) // 2] for k, v in by_cross.items()}
    ks = sorted(typical)
    for k0, k1 in zip(ks, ks[1:]):
        assert typical[k1] < typical[k0], typical
    for k, v in by_cross.items():
        assert typical[k] >= 0.9 * max(v)


def test_no_packed_groups_means_no_stream_ctas(vc):
    s = vc.shape(4, 64, 8, 128, bits=2)
    n, lo, max_parts = vc.vc_draft_attn_partition(s, 0, 152)
    assert (n, lo, max_parts) == (0, [0], 1)


def test_partition_argument_errors(vc):
    s = vc.shape(4, 64, 8, 128, bits=2)
    for mp, slots in [(33, 152), (-32, 152), (1024, 0)]:
        with pytest.raises(vc.VcError) as e:
            vc.vc_draft_attn_partition(s, mp, slots)
        assert e.value.status == 1
