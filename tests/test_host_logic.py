"""Host-side logic without a GPU: replica reduction over 2 gloo ranks, the
bench's rank arithmetic, host fault injection, and the reference arm's
bookkeeping."""
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_setup()
    bench.dist_barrier(w)
    # rank r processed (r + 1) * 1000 tokens in (r + 1) * 10 ms
    value = ((r + 1) * 1000) / ((r + 1) * 10 / 1e3)
    out = bench.reduce_over_ranks(value, 50.0 * (r + 1), (r + 1) * 10.0, w)
    q.put((r, out))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replica_reduction_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    # all tokens (1000 + 2000) over the slowest rank's 20 ms; e2e adds; max time
    for r in range(2):
        value, e2e, t = res[r]
        assert t == 20.0
        assert value == pytest.approx(3000 / 0.020)
        assert e2e == pytest.approx(150.0)


def test_combine_rank_results_single():
    import bench
    assert bench.combine_rank_results([(5.0, 4.0, 2.0)]) == (5.0, 4.0, 2.0)


def test_injected_h2d_failure_returns_status_without_a_gpu(monkeypatch):
    from verify_compressed_kv_gb300 import _lib as vc
    monkeypatch.setenv("VC_FAULT", "h2d_fail")
    s = vc.shape(1, 4, 1, 64, k=1)
    # all pointers non-NULL (plain integers): the call must fail on the injected fault
    with pytest.raises(vc.VcError) as e:
        vc.vc_verify_attn_streamed(0x1000, s, 0x2000, 0x3000, 64, 64, 64, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 1,
                                   0x9000, 1 << 30, 0, 0)
    assert e.value.status == 3 and "injected" in str(e.value)


def test_streamed_rejects_a_prefix_past_the_store():
    """max_prefix beyond the pinned store's capacity is an argument error (checked
    on the host, before any copy could read past the store)."""
    from verify_compressed_kv_gb300 import _lib as vc
    s = vc.shape(1, 4, 1, 64, k=1)
    with pytest.raises(vc.VcError) as e:
        vc.vc_verify_attn_streamed(0x1000, s, 0x2000, 0x3000, 64, 128 + 1, 128, 0x4000, 0x5000, 0x6000, 0x7000,
                                   0x8000, 1, 0x9000, 1 << 30, 0, 0)
    assert e.value.status == 1 and "outside the store" in str(e.value)
    with pytest.raises(vc.VcError) as e:
        vc.vc_verify_prefetch(0x1000, s, 0x3000, 64, 65, 64, 0x5000, 0)
    assert e.value.status == 1
    with pytest.raises(vc.VcError) as e:
        vc.vc_verify_prefetch(0x1000, s, 0x3000, 64, 10, 100, 0x5000, 0)      # capacity not a multiple of C
    assert e.value.status == 1


def test_workload_table_matches_the_shapes():
    import synth
    w = synth.get("mistral")
    assert (w.B, w.Hq, w.Hkv, w.d, w.T, w.k, w.bits, w.V, w.C) == (8, 32, 8, 128, 32768, 16, 2, 32768, 4096)
    q = synth.get("qwen")
    assert q.T_keep == 16384 and q.bits == 4 and q.G == 5
    ll = synth.get("llama")
    assert ll.layers == 8 and ll.G == 8 and ll.T == 131072
    st = synth.get("stagger")
    assert st.groups == 2 and st.B == 32 and st.k == 24


def test_length_bounds_are_the_longest_request_not_a_sum_of_maxima():
    """The host bounds the drafting and the full-KV transfer use: max_prefix is
    the longest request's prefix (prefix at load + its own committed tokens,
    n_acc + 1 a round), not the sum of each round's largest commit;
    max_packed follows the same tokens from the packed length at load."""
    from verify_compressed_kv_gb300.runtime import LengthBounds
    b = LengthBounds(3)
    b.prefix_from(1000)
    b.packed_from(992)
    assert (b.max_prefix, b.max_packed) == (1000, 992)
    b.commit([5, 0, 2])                      # commits 6, 1, 3
    assert (b.max_prefix, b.max_packed) == (1006, 998)
    b.commit([0, 9, 2])                      # totals 7, 11, 6: the sum of maxima would say 16
    assert (b.max_prefix, b.max_packed) == (1011, 1003)
    b.commit([0, 0, 0])
    assert b.max_prefix == 1012
    b.prefix_from(2048)                      # a new prefix: commits counted from there
    b.packed_from(512)                       # e.g. the kept tokens of a token-dropped prefix
    assert (b.max_prefix, b.max_packed) == (2048, 512)
    b.commit([31, 3, 0])
    assert (b.max_prefix, b.max_packed) == (2080, 544)
