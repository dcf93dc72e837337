"""The allocation-free accept entry point (vc_accept_noalloc).

It serves callers that cannot allocate device memory (a plugin given only its
input and output buffers by a framework that owns all device memory, or a
loop where cudaMalloc's possible device synchronisation is not allowed).  Its
results must equal those of vc_accept with a caller-provided workspace, on
two calls in a row (the fixed scratch keeps the previous call's contents).
This file is collected last, so a failure here stops a run only after every
other test has run.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import accept as oacc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    from verify_compressed_kv_gb300 import _lib
    return _lib


def _run_both(vc, logits, drafts):
    B, R, V = logits.shape
    k = R - 1
    lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    dr = torch.from_numpy(np.ascontiguousarray(drafts, np.int32)).cuda()
    outs = []
    for fn in ("ws", "noalloc"):
        n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        am = torch.full((B, R), -1, dtype=torch.int32, device="cuda")
        if fn == "ws":
            wsb = vc.vc_accept_workspace_size(B, k, V)
            ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
            vc.vc_accept(B, k, V, lg, dr, n, nxt, am, ws, wsb)
        else:
            vc.vc_accept_noalloc(B, k, V, lg, dr, n, nxt, am)
        torch.cuda.synchronize()
        outs.append((n.cpu().numpy(), nxt.cpu().numpy(), am.cpu().numpy()))
    return outs


@pytest.mark.parametrize("name", ["mistral", "tiny"])
def test_noalloc_matches_workspace_entry_point_twice(vc, name):
    w = synth.get(name)
    for rnd in range(2):                         # two calls in a row on the shared scratch
        logits, drafts, _ = synth.logits_and_drafts(w, rnd)
        (n0, x0, a0), (n1, x1, a1) = _run_both(vc, logits, drafts)
        assert np.array_equal(n0, n1) and np.array_equal(x0, x1) and np.array_equal(a0, a1)
        on, ox, oa = oacc.accept(logits, drafts)
        assert np.array_equal(n1, on) and np.array_equal(x1, ox) and np.array_equal(a1, oa)


def test_noalloc_ties_and_small_vocab(vc):
    rng = np.random.default_rng(5)
    for V in (7, 1001):
        logits = rng.integers(-3, 4, size=(6, 5, V)).astype(np.float32)
        drafts = rng.integers(0, V, size=(6, 4)).astype(np.int32)
        (n0, x0, a0), (n1, x1, a1) = _run_both(vc, logits, drafts)
        assert np.array_equal(n0, n1) and np.array_equal(x0, x1) and np.array_equal(a0, a1)
        on, ox, oa = oacc.accept(logits, drafts)
        assert np.array_equal(n1, on) and np.array_equal(x1, ox) and np.array_equal(a1, oa)


def test_noalloc_rejects_sizes_beyond_its_scratch(vc):
    B, k, V = 200, 40, 64          # B*(k+1) = 8200 rows > 6144 partials
    lg = torch.zeros((B, k + 1, V), dtype=torch.float32, device="cuda")
    dr = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    o = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(vc.VcError) as e:
        vc.vc_accept_noalloc(B, k, V, lg, dr, o, o, None)
    assert e.value.status == 6 and "scratch limit" in str(e.value)


def test_noalloc_rejects_more_requests_than_its_counters(vc):
    B, k, V = 4097, 0, 1           # one row per request: 4097 partials fit, 4097 counters do not
    lg = torch.zeros((B, k + 1, V), dtype=torch.float32, device="cuda")
    o = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(vc.VcError) as e:
        vc.vc_accept_noalloc(B, k, V, lg, None, o, o, None)
    assert e.value.status == 6 and "4096 requests" in str(e.value)
